// Host-side cache of per-device launch facts: SM counts, occupancy-derived
// grid caps, kernel attributes already set, device addresses of the library's
// __device__ symbols. Each value is tagged with the CUDA context it was
// looked up in, so a context created later on the same device (after
// cudaDeviceReset, or a context the caller made current) looks it up again
// instead of reusing an address or setting that belongs to a destroyed one.
#pragma once

#include <mutex>

#include <cuda_runtime.h>

namespace bea {

constexpr int kMaxCachedDevices = 64;

// Unique id (cuCtxGetId) of the calling thread's current context; 0 when no
// context is current yet or the driver entry points cannot be found, in which
// case callers do not cache.
unsigned long long current_context_id();

// One value of type T per device, valid for the context it was computed in.
template <typename T>
class PerContext {
 public:
  // *out = the cached value for the current device and context, or
  // compute(&value) when there is none (cached on success).
  template <typename F>
  cudaError_t get(F compute, T* out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long ctx = current_context_id();
    const bool cacheable = ctx != 0 && dev >= 0 && dev < kMaxCachedDevices;
    if (cacheable) {
      std::lock_guard<std::mutex> lock(mutex_);
      if (ctx_[dev] == ctx) {
        *out = value_[dev];
        return cudaSuccess;
      }
    }
    T v{};
    e = compute(&v);
    if (e != cudaSuccess) return e;
    if (cacheable) {
      std::lock_guard<std::mutex> lock(mutex_);
      ctx_[dev] = ctx;
      value_[dev] = v;
    }
    *out = v;
    return cudaSuccess;
  }

 private:
  std::mutex mutex_;
  unsigned long long ctx_[kMaxCachedDevices] = {};
  T value_[kMaxCachedDevices] = {};
};

// SM count of the current device (cached per context).
cudaError_t device_sm_count(int* sms);

// One wave of resident CTAs of `kern` at `threads` threads and `smem` bytes of
// dynamic shared memory: SM count x CTAs per SM (at least 1 per SM).
template <typename K>
cudaError_t wave_cap(PerContext<int>& cache, K kern, int threads, size_t smem, int* cap) {
  return cache.get(
      [&](int* v) {
        int sms = 0, per_sm = 0;
        cudaError_t e = device_sm_count(&sms);
        if (e != cudaSuccess) return e;
        if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, smem)) != cudaSuccess)
          return e;
        *v = sms * (per_sm > 0 ? per_sm : 1);
        return cudaSuccess;
      },
      cap);
}

}  // namespace bea
