// device.h -- per-device facts and one-time set-up for the launch planners (host code).
//
// The planners size grids and pipelines from the device they launch on: SM count and
// shared memory per SM / per block are queried once per device ordinal (attribute reads,
// not driver calls on every launch), and kernel attributes such as the shared-memory
// opt-in are set once per device, since they are per-device state of the function.
#pragma once

#include <cuda_runtime.h>

#include <mutex>

namespace moe {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  int ordinal;
  int sms;                // multiprocessors
  size_t smem_per_sm;     // shared memory per multiprocessor (bytes)
  size_t smem_optin;      // largest dynamic shared memory a block can opt in to (bytes)
};

// Facts of the current device (cached per ordinal). sms == 0 if the query failed.
inline DeviceInfo device_info() {
  static std::mutex mu;
  static DeviceInfo cache[kMaxDevices];
  static bool have[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DeviceInfo{-1, 0, 0, 0};
  std::lock_guard<std::mutex> lock(mu);
  if (!have[dev]) {
    int sms = 0, per_sm = 0, optin = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
      return DeviceInfo{dev, 0, 0, 0};
    cache[dev] = DeviceInfo{dev, sms, (size_t)per_sm, (size_t)optin};
    have[dev] = true;
  }
  return cache[dev];
}

// Run `fn` once per device ordinal (with that device current).
struct PerDeviceOnce {
  std::mutex mu;
  bool done[kMaxDevices] = {};
};
template <class F>
inline void once_per_device(PerDeviceOnce& o, F&& fn) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return;
  std::lock_guard<std::mutex> lock(o.mu);
  if (!o.done[dev]) {
    fn();
    o.done[dev] = true;
  }
}

}  // namespace moe
