// host_util.h -- small host-side helpers shared by the C ABI translation
// units (api.cu, stack_api.cu): CUDA error mapping, host<->device copies,
// alignment and overlap checks.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "prnn.h"

namespace prnn {

inline prnn_status_t cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return PRNN_OK;
  if (e == cudaErrorMemoryAllocation) return PRNN_ERR_OOM;
  if (e == cudaErrorCooperativeLaunchTooLarge) return PRNN_ERR_UNSUPPORTED;
  return PRNN_ERR_CUDA;
}

#define PRNN_TRY(expr)                                  \
  do {                                                  \
    cudaError_t e_ = (expr);                            \
    if (e_ != cudaSuccess) return cuda_status(e_);      \
  } while (0)

template <typename T>
inline void free_dev(T*& p) {
  if (p) cudaFree((void*)p);
  p = nullptr;
}

// Copy n bytes from any CUDA-readable pointer (device, managed, host) to host.
inline cudaError_t to_host(void* dst, const void* src, size_t n) {
  return cudaMemcpy(dst, src, n, cudaMemcpyDefault);
}

template <typename T>
inline cudaError_t upload(T** dptr, const void* src, size_t bytes) {
  T* p = nullptr;
  cudaError_t e = cudaMalloc((void**)&p, bytes ? bytes : 16);
  if (e != cudaSuccess) return e;
  e = cudaMemcpy(p, src, bytes, cudaMemcpyHostToDevice);
  if (e != cudaSuccess) {
    cudaFree(p);
    return e;
  }
  *dptr = p;
  return cudaSuccess;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const char* pa = static_cast<const char*>(a);
  const char* pb = static_cast<const char*>(b);
  return pa < pb + nb && pb < pa + na;
}

inline int round_up(int v, int m) { return (v + m - 1) / m * m; }

}  // namespace prnn
