// per_device.h -- host-side state that CUDA keeps per device: a kernel's
// dynamic shared-memory limit (cudaFuncSetAttribute) and values derived from
// it, such as the number of resident CTA pairs.  Each is set up once per
// device, under a lock, the first time a launch reaches that device.
#pragma once

#include <cuda_runtime.h>

#include <mutex>

namespace gbmoe {

constexpr int kMaxDevices = 64;

// The device current on the calling thread, or -1 when there is none or its
// ordinal is beyond the table.
inline int current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
  return dev;
}

// One int per device, filled by `make` (returning a cudaError_t and writing
// the value) the first time it is asked for on that device.
struct PerDeviceInt {
  std::mutex mu;
  bool ready[kMaxDevices] = {};
  int value[kMaxDevices] = {};

  template <class Make>
  cudaError_t get(int *out, Make make) {
    const int dev = current_device();
    if (dev < 0) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(mu);
    if (!ready[dev]) {
      int v = 0;
      cudaError_t e = make(&v);
      if (e != cudaSuccess) return e;
      value[dev] = v;
      ready[dev] = true;
    }
    *out = value[dev];
    return cudaSuccess;
  }
};

// cudaFuncSetAttribute(kernel, MaxDynamicSharedMemorySize, bytes) once per
// device for this kernel.
template <class Kernel>
cudaError_t set_smem_once(PerDeviceInt &flag, Kernel kernel, int bytes) {
  int unused = 0;
  return flag.get(&unused, [&](int *v) {
    *v = bytes;
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  });
}

}  // namespace gbmoe
