// Host-side helpers shared by the entry points (validation, launch checks,
// per-device launch geometry).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "eagle.h"

namespace eagle {

#define EAGLE_CHECK_ARG(cond)                   \
  do {                                          \
    if (!(cond)) return EAGLE_ERR_INVALID_ARG;  \
  } while (0)

#define EAGLE_CHECK_SHAPE(cond)                      \
  do {                                               \
    if (!(cond)) return EAGLE_ERR_UNSUPPORTED_SHAPE; \
  } while (0)

#define EAGLE_CUDA(call)                          \
  do {                                            \
    if ((call) != cudaSuccess) {                  \
      (void)cudaGetLastError();                   \
      return EAGLE_ERR_CUDA;                      \
    }                                             \
  } while (0)

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline eagle_status launch_status() {
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? EAGLE_OK : EAGLE_ERR_CUDA;
}

// Number of SMs of the current device (queried per call; cheap attribute read).
inline int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

}  // namespace eagle
