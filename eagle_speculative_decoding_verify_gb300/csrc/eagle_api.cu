// Library-wide entry points: status strings, version, workspace helpers.
#include "eagle_common.cuh"
#include "eagle_host.h"

using namespace eagle;

extern "C" const char* eagle_status_string(eagle_status s) {
  switch (s) {
    case EAGLE_OK: return "ok";
    case EAGLE_ERR_INVALID_ARG: return "invalid argument";
    case EAGLE_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case EAGLE_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case EAGLE_ERR_CUDA: return "CUDA error";
    case EAGLE_ERR_TIMEOUT: return "device wait timed out";
    case EAGLE_ERR_DEVICE_ASSERT: return "device invariant violated";
  }
  return "unknown status";
}

extern "C" int32_t eagle_version(void) { return 2; }

#ifndef EAGLE_BUILD_ID
#define EAGLE_BUILD_ID "unknown"
#endif

// Hash of the sources and flags this library was compiled from (set by the
// build script), so that a caller can tell a stale binary from a current one.
extern "C" const char* eagle_build_id(void) { return EAGLE_BUILD_ID; }

extern "C" eagle_status eagle_workspace_init(void* ws, size_t ws_bytes, eagle_stream stream) {
  EAGLE_CHECK_ARG(ws != nullptr && ws_bytes >= kWsHeader);
  EAGLE_CUDA(cudaMemsetAsync(ws, 0, ws_bytes, reinterpret_cast<cudaStream_t>(stream)));
  return EAGLE_OK;
}

extern "C" eagle_status eagle_workspace_error(const void* ws, eagle_stream stream,
                                              int32_t* status, int32_t* detail) {
  EAGLE_CHECK_ARG(ws != nullptr && status != nullptr);
  int32_t h[2] = {0, 0};
  EAGLE_CUDA(cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)));
  EAGLE_CUDA(cudaMemcpy(h, ws, sizeof(h), cudaMemcpyDeviceToHost));
  *status = h[0];
  if (detail) *detail = h[1];
  return EAGLE_OK;
}
