// Host-side helpers shared by the launchers: per-device one-time set-up that
// is safe when several host threads make their first call at the same time,
// the device's SM count, and the driver's tensor-map encoder.
#pragma once

#include <atomic>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <mutex>

namespace csa2 {

constexpr int MAX_DEVICES = 64;

// Runs a set-up function once per device, with that device current.  The
// first caller on a device runs it under a lock; concurrent callers wait for
// it; later callers see the result with one atomic load.  A failed set-up is
// not recorded, so the next call tries again.  Objects of this type must have
// static storage duration (their flags start at zero).
class PerDeviceOnce {
 public:
  template <class F>
  cudaError_t ensure(F&& init) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= MAX_DEVICES) return cudaErrorInvalidDevice;
    if (done_[dev].load(std::memory_order_acquire)) return cudaSuccess;
    std::lock_guard<std::mutex> lock(mu_);
    if (done_[dev].load(std::memory_order_relaxed)) return cudaSuccess;
    e = init(dev);
    if (e == cudaSuccess) done_[dev].store(1, std::memory_order_release);
    return e;
  }

 private:
  std::mutex mu_;
  std::atomic<int> done_[MAX_DEVICES];
};

// Number of SMs of the current device (queried once per device).
inline cudaError_t device_sms(int* n) {
  static PerDeviceOnce once;
  static int sms[MAX_DEVICES];
  int dev = 0;
  cudaError_t e = once.ensure([&](int d) {
    int v = 0;
    cudaError_t r = cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, d);
    if (r == cudaSuccess && v <= 0) r = cudaErrorInvalidDevice;
    if (r == cudaSuccess) sms[d] = v;
    return r;
  });
  if (e != cudaSuccess) return e;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  *n = sms[dev];
  return cudaSuccess;
}

// cuTensorMapEncodeTiled from the driver, looked up once per process
// (initialisation of a function-local static is thread safe); null if missing.
inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
  }();
  return fn;
}

}  // namespace csa2
