// Host-side, per-device one-time set-up (function attributes, symbol
// addresses).
//
// Kernel function attributes (the dynamic shared-memory limit, the carveout)
// and the device address of a __device__ array belong to one device's
// context: a launch on a second device needs them set there too, and a
// context that was reset (cudaDeviceReset) and created again has lost them.
// DeviceOnce remembers, per device, the id of the context in which the set-up
// last succeeded, so it runs again on a new device or in a new context.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

namespace tf {

constexpr int kMaxDevices = 64;

// Unique id of the calling thread's current CUDA context (0 if none or not
// available).  Driver entry points are looked up through the runtime, so the
// library links only against cudart.
inline uint64_t current_context_id() {
  using GetCurrent = CUresult (*)(CUcontext*);
  using GetId = CUresult (*)(CUcontext, unsigned long long*);
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrent>(f);
    else
      (void)cudaGetLastError();
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetId>(f);
    else
      (void)cudaGetLastError();
  });
  if (!get_current || !get_id) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return static_cast<uint64_t>(id);
}

struct DeviceOnce {
  std::mutex mu;
  uint64_t ctx[kMaxDevices] = {};  // context id of the last successful set-up, 0 = none
};

// Runs fn() unless it already succeeded on the current device in its current
// context.  fn returns a cudaError_t; a failure is returned and retried on
// the next call.
template <typename Fn>
cudaError_t device_once(DeviceOnce& o, Fn fn) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return fn();
  std::lock_guard<std::mutex> lock(o.mu);
  const uint64_t id = current_context_id();
  if (id != 0 && o.ctx[dev] == id) return cudaSuccess;
  e = fn();
  if (e == cudaSuccess) o.ctx[dev] = current_context_id();
  return e;
}

}  // namespace tf
