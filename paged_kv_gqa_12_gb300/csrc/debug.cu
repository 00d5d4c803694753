// pa_debug_wait_expiry: one bounded device-side wait run out on purpose, so
// that a test can check the expiry path of the waits every kernel of the
// library uses -- the error bit they set, that they return, and that a CTA
// whose peers already recorded an expired wait gives up at once instead of
// waiting out its own limit.
//
// The kernel is one CTA of one warp with no TMA copy, tensor-core operation or
// memory traffic of any other kind in flight: lane 0 initialises an mbarrier
// that nothing ever arrives on and waits for its first phase through one of
// the shared wait helpers with a short limit.  Every helper measures the limit
// on %globaltimer, so the wait ends by itself.
#include <cstdint>

#include <cuda_runtime.h>

#include "pa.h"
#include "pa_internal.h"
#include "ptx.cuh"

namespace pa {
namespace {

constexpr int64_t kResultOffset = 64;   // inside the scratch header, clear of the error word and counters

__global__ void __launch_bounds__(32) wait_expiry_kernel(uint32_t* err, int64_t* result, int which,
                                                          uint64_t limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  fence_mbar_init();
  if (which >= 3) atomicOr(err, kErrWaitTimeout);   // another CTA's wait already expired
  const uint64_t t0 = globaltimer_ns();
  bool ok;
  switch (which) {
    case 0: ok = mbar_wait(&bar, 0, err, limit_ns); break;
    case 1:
    case 3: ok = wait_or_abort(&bar, 0, err, limit_ns); break;
    default: ok = poll_or_abort(&bar, 0, err, limit_ns); break;
  }
  result[0] = ok ? 1 : 0;
  result[1] = static_cast<int64_t>(globaltimer_ns() - t0);
}

}  // namespace
}  // namespace pa

extern "C" pa_status pa_debug_wait_expiry(void* scratch, int32_t which, int64_t limit_ns, void* stream) {
  if (!scratch || which < 0 || which > 4) return PA_ERR_INVALID_ARG;
  if (limit_ns < 1000 || limit_ns > 100000000) return PA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(scratch) & 255u) != 0) return PA_ERR_UNSUPPORTED;
  uint8_t* sc = static_cast<uint8_t*>(scratch);
  pa::wait_expiry_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      reinterpret_cast<uint32_t*>(sc), reinterpret_cast<int64_t*>(sc + pa::kResultOffset), which,
      static_cast<uint64_t>(limit_ns));
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}
