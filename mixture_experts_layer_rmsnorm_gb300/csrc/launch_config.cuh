// launch_config.cuh -- host-side configuration of a kernel that is done once
// per device (function attributes, occupancy queries) and is safe to reach from
// several host threads: each launcher keeps a function-local PerDevice.
#pragma once

#include <cuda_runtime.h>

#include <mutex>

namespace moe {

constexpr int kMaxDevices = 64;

// The result of `make(value)` for the current device, computed on the first
// call for that device; `make` returns the configuration's status and may set
// an int (e.g. an occupancy figure), returned through `out`.
struct PerDevice {
  std::once_flag once[kMaxDevices];
  cudaError_t status[kMaxDevices] = {};
  int value[kMaxDevices] = {};

  template <typename F>
  cudaError_t get(F&& make, int* out = nullptr) {
    int dev = 0;
    const cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::call_once(once[dev], [&] { status[dev] = make(value[dev]); });
    if (out) *out = value[dev];
    return status[dev];
  }
};

}  // namespace moe
