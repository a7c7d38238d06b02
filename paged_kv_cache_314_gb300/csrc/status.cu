// status.cu -- ABI version and status strings.
#include "pa.h"

extern "C" int pa_abi_version(void) { return 1; }

extern "C" const char* pa_status_string(pa_status status) {
    switch (status) {
        case PA_OK: return "ok";
        case PA_ERR_INVALID_ARG: return "invalid argument";
        case PA_ERR_UNSUPPORTED: return "unsupported shape or type";
        case PA_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
        case PA_ERR_CUDA: return "CUDA error";
    }
    return "unknown status";
}
