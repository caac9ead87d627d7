// Version and status strings of the C ABI declared in include/pa.h, and the
// read-back of a device error word.
#include <cuda_runtime.h>

#include "../../include/pa.h"

extern "C" int32_t pa_abi_version(void) { return PA_ABI_VERSION; }

extern "C" const char *pa_status_string(pa_status status) {
  switch (status) {
    case PA_OK: return "ok";
    case PA_ERR_INVALID_ARG: return "invalid argument";
    case PA_ERR_UNSUPPORTED: return "unsupported shape";
    case PA_ERR_WORKSPACE: return "workspace missing or too small";
    case PA_ERR_LAUNCH: return "kernel launch failed";
    case PA_ERR_DEVICE: return "device query failed";
    default: return "unknown status";
  }
}

extern "C" pa_status pa_get_device_error(int32_t *error_word, int32_t *out_flags, int32_t clear,
                                         void *stream) {
  if (!error_word || !out_flags) return PA_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t host = 0;
  if (cudaMemcpyAsync(&host, error_word, sizeof host, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return PA_ERR_DEVICE;
  if (clear && cudaMemsetAsync(error_word, 0, sizeof(int32_t), s) != cudaSuccess)
    return PA_ERR_DEVICE;
  if (cudaStreamSynchronize(s) != cudaSuccess) return PA_ERR_DEVICE;
  *out_flags = host;
  return PA_OK;
}
