// Host helpers shared by the kernels' launchers: the driver's tensor-map
// encoder, fetched once through the runtime (no link against libcuda), and a
// per-device cache of occupancy figures.  Both are safe to use from several
// host threads at once.
#pragma once

#include <atomic>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

namespace fp8bs {

inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  // initialised exactly once, even with concurrent first calls
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    return nullptr;
  }();
  return fn;
}

constexpr int kMaxCachedDevices = 64;

// An occupancy figure of one kernel configuration on the current device,
// computed by `query(&value)` on first use per device and cached (a value of
// at least 1 is stored; concurrent first uses may both query, with the same
// result).
template <typename Query>
cudaError_t cached_per_device(std::atomic<int> (&cache)[kMaxCachedDevices], Query query, int* value) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < kMaxCachedDevices) {
    const int v = cache[dev].load(std::memory_order_relaxed);
    if (v > 0) {
      *value = v;
      return cudaSuccess;
    }
  }
  int n = 0;
  e = query(&n);
  if (e != cudaSuccess) return e;
  n = n > 0 ? n : 1;
  if (dev >= 0 && dev < kMaxCachedDevices) cache[dev].store(n, std::memory_order_relaxed);
  *value = n;
  return cudaSuccess;
}

}  // namespace fp8bs
