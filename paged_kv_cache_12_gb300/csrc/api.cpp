// Status text, version and the debug-validation switch of libpa.
#include <cstdlib>
#include <cstring>

#include "pa.h"

namespace pa {

bool debug_validate() {
    static const bool on = [] {
        const char *v = std::getenv("PA_DEBUG_VALIDATE");
        return v && std::strcmp(v, "0") != 0 && v[0] != '\0';
    }();
    return on;
}

}  // namespace pa

extern "C" const char *pa_status_string(int status) {
    switch (status) {
    case PA_OK: return "ok";
    case PA_ERR_INVALID_ARG: return "invalid argument";
    case PA_ERR_OUT_OF_BLOCKS: return "out of blocks: the free queue cannot cover the request";
    case PA_ERR_STATE: return "allocator state inconsistent";
    case PA_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case PA_ERR_CUDA: return "CUDA runtime error";
    case PA_ERR_UNSUPPORTED: return "unsupported head_dim, block_size or group size";
    case PA_ERR_TIMEOUT: return "a kernel timed out waiting for its own copies";
    default: return "unknown status";
    }
}

extern "C" int pa_version(void) { return 1; }
