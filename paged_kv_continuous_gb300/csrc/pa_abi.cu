// Version and status strings of the C ABI declared in include/pa.h.
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
