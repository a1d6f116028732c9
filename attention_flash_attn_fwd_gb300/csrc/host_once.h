// host_once.h -- one-time host set-up of a kernel, per device.
//
// Function attributes such as the dynamic shared-memory limit are set per
// device, so a single process-wide "configured" flag would skip the set-up on
// the second device a process uses and that device's launch would fail.
#pragma once

#include <cuda_runtime.h>

#include <atomic>

namespace attn_host {

// Runs `setup` for the current device until it has succeeded once there and
// returns its error otherwise.  Threads racing on the first call may each run
// it; `setup` must be idempotent (cudaFuncSetAttribute and
// cudaFuncGetAttributes are).  Devices past the 64th run it on every call.
template <typename F>
inline cudaError_t once_per_device(std::atomic<unsigned long long>& done, F&& setup) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
  if (bit != 0ull && (done.load(std::memory_order_acquire) & bit) != 0ull) return cudaSuccess;
  e = setup();
  if (e == cudaSuccess && bit != 0ull) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

}  // namespace attn_host
