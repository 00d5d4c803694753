// Decode with a library-owned workspace: pa_decode_static_scratch.
//
// Some callers cannot hand the library a scratch buffer: code that runs where
// it may not allocate device memory (a host runtime or plugin without a device
// allocator, or a process whose memory pool already owns the whole GPU), or
// code that must never allocate so that its latency stays fixed.  For them this
// entry point runs the ordinary decode kernels with the split-KV workspace taken
// from a fixed array that lives in this library's device image.
//
// The array is kStaticScratchBytes (16 MiB) on every GPU that loads the
// library, held until the process exits.  Plans whose scratch_bytes exceed it
// are rejected.  All calls on a device share the one array, which keeps the
// previous call's contents; calls that overlap on the GPU (different streams,
// or different host threads) race on it and must be serialised by the caller.
#include <mutex>

#include <cuda_runtime.h>

#include "pa.h"
#include "pa_internal.h"

namespace pa {
namespace {

constexpr int64_t kStaticScratchBytes = int64_t{16} << 20;
constexpr int kMaxDevices = 256;

static __device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_decode_scratch on the current device.  In host code the
// array's name is only a host-side handle, so the address must come from the
// runtime.  It is looked up again on every call made outside a stream capture
// (a device reset reloads the library's module, possibly elsewhere); a call
// being captured uses the address found by the last uncaptured call on that
// device, and fails if there was none.
pa_status static_scratch(cudaStream_t stream, void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PA_ERR_CUDA;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) return PA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (cap == cudaStreamCaptureStatusNone) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr) return PA_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  if (!g_scratch_ptr[dev]) return PA_ERR_CUDA;
  *out = g_scratch_ptr[dev];
  return PA_OK;
}

}  // namespace
}  // namespace pa

extern "C" pa_status pa_decode_static_scratch(
    const pa_plan_t* plan, const void* q, int64_t q_stride_tok, int64_t q_stride_head, const void* k_cache,
    const void* v_cache, int64_t kv_stride_page, int64_t kv_stride_tok, int64_t kv_stride_head, int32_t num_pages,
    const int32_t* block_table, int64_t bt_stride, const int32_t* seq_lens, int32_t batch, float scale,
    const float* sinks, float k_scale, float v_scale, void* out, int64_t out_stride_tok, int64_t out_stride_head,
    float* lse, void* stream) {
  if (!plan) return PA_ERR_INVALID_ARG;
  if (plan->scratch_bytes > pa::kStaticScratchBytes) return PA_ERR_SCRATCH_TOO_SMALL;
  void* scratch = nullptr;
  const pa_status st = pa::static_scratch(static_cast<cudaStream_t>(stream), &scratch);
  if (st != PA_OK) return st;
  // The header (error word, split-arrival counters) must start at zero; the
  // split partials behind it are always written before they are read.
  if (cudaMemsetAsync(scratch, 0, pa::kScratchHeaderBytes, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return PA_ERR_CUDA;
  return pa_decode(plan, q, q_stride_tok, q_stride_head, k_cache, v_cache, kv_stride_page, kv_stride_tok,
                   kv_stride_head, num_pages, block_table, bt_stride, seq_lens, batch, scale, sinks, k_scale,
                   v_scale, nullptr, nullptr, out, out_stride_tok, out_stride_head, lse, scratch,
                   pa::kStaticScratchBytes, stream);
}
