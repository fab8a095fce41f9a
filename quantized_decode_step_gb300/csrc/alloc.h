// Allocation through one place, so that a test can make chosen allocations fail on the host
// (mag_debug_fail_allocations) without any fault on the device.
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>

namespace mag {

// True when the allocation about to be made is to fail (consumes one injected failure).
bool alloc_injected_failure();

inline cudaError_t dev_malloc(void** p, size_t bytes) {
  if (alloc_injected_failure()) return cudaErrorMemoryAllocation;
  return cudaMalloc(p, bytes);
}
template <typename T>
inline cudaError_t dev_malloc(T** p, size_t bytes) {
  return dev_malloc(reinterpret_cast<void**>(p), bytes);
}
inline cudaError_t dev_malloc_async(void** p, size_t bytes, cudaStream_t s) {
  if (alloc_injected_failure()) return cudaErrorMemoryAllocation;
  return cudaMallocAsync(p, bytes, s);
}
inline cudaError_t host_alloc(void** p, size_t bytes, unsigned flags) {
  if (alloc_injected_failure()) return cudaErrorMemoryAllocation;
  return cudaHostAlloc(p, bytes, flags);
}
template <typename T>
inline cudaError_t host_alloc(T** p, size_t bytes, unsigned flags) {
  return host_alloc(reinterpret_cast<void**>(p), bytes, flags);
}

}  // namespace mag
