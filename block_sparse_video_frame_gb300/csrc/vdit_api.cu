// Error reporting and version of libvdit.
#include <cstdarg>
#include <cstdio>

#include "vdit_internal.h"

namespace vdit {

namespace {
thread_local char g_err[512] = "";
}

void set_error(const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
}

void clear_error() { g_err[0] = '\0'; }

vdit_status cuda_fail(cudaError_t e, const char *what) {
    set_error("%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
    return VDIT_ERR_CUDA;
}

}  // namespace vdit

extern "C" const char *vdit_last_error(void) { return vdit::g_err; }

extern "C" const char *vdit_version(void) { return "libvdit 0.1 (sm_103a, tcgen05)"; }
