// Error reporting and version of libvdit.
#include <atomic>
#include <cstdarg>
#include <cstdio>

#include "vdit_internal.h"

namespace vdit {

namespace {
thread_local char g_err[512] = "";
std::atomic<unsigned long long> g_wait_limit_ns{kDefaultWaitLimitNs};
}

unsigned long long wait_limit_ns() { return g_wait_limit_ns.load(std::memory_order_relaxed); }

namespace {
std::atomic<int> g_fail_after{0};   // > 0: allocations left until the one that fails
}

cudaError_t device_alloc(void **ptr, size_t bytes) {
    int n = g_fail_after.load(std::memory_order_relaxed);
    while (n > 0) {
        if (g_fail_after.compare_exchange_weak(n, n - 1, std::memory_order_relaxed)) {
            if (n == 1) {
                *ptr = nullptr;
                return cudaErrorMemoryAllocation;
            }
            break;
        }
    }
    return cudaMalloc(ptr, bytes);
}

namespace {
std::atomic<int> g_launch_fail_after{0};   // > 0: attention launches left until the one that fails
}

bool launch_fails_by_hook() {
    int n = g_launch_fail_after.load(std::memory_order_relaxed);
    while (n > 0) {
        if (g_launch_fail_after.compare_exchange_weak(n, n - 1, std::memory_order_relaxed))
            return n == 1;
    }
    return false;
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

extern "C" void vdit_set_wait_limit_ns(uint64_t ns) {
    vdit::g_wait_limit_ns.store(ns == 0 ? vdit::kDefaultWaitLimitNs : ns, std::memory_order_relaxed);
}

extern "C" void vdit_set_alloc_fail_after(int32_t n) {
    vdit::g_fail_after.store(n > 0 ? n : 0, std::memory_order_relaxed);
}

extern "C" void vdit_set_launch_fail_after(int32_t n) {
    vdit::g_launch_fail_after.store(n > 0 ? n : 0, std::memory_order_relaxed);
}

extern "C" const char *vdit_version(void) { return "libvdit 0.1 (sm_103a, tcgen05)"; }
