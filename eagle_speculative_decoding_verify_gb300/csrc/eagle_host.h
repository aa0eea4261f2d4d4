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

// Launch attribute that lets the kernel start before the previous kernel in
// the stream has completed (programmatic dependent launch); the row-stream
// kernels (build, verify, per-depth build, policies), the tree finalisation
// and the KV commit use it.  Every kernel launched with it calls pdl_wait()
// before it reads or writes anything the previous kernels may produce or use;
// only work on the library's own static scratch (code warm-ups) and on-chip
// set-up run before that.  Every kernel of the library calls pdl_trigger() at
// its start: the next kernel's CTAs then launch once every CTA of this grid
// has triggered or exited -- so all of this grid's CTAs are already running
// and the waiting ones can never hold an SM this grid still needs.  (The
// attention kernels themselves are launched without the attribute: measured,
// their early CTAs lengthened the step.)
inline void pdl_attribute(cudaLaunchAttribute& a) {
  a.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  a.val.programmaticStreamSerializationAllowed = 1;
}

// kernel<<<grid, block, smem, stream>>>(args...) with pdl_attribute.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  pdl_attribute(attr[0]);
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Number of SMs of the current device (queried per call; cheap attribute read).
inline int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

}  // namespace eagle
