// api.cu -- library-wide entry points: version, status strings, error detail, and the
// per-device property cache used to size grids.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdarg>
#include <cstdio>

#include "sd_host.h"

namespace sd {

static thread_local char g_err[512];

void set_error(const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
}

void clear_error() { g_err[0] = '\0'; }

namespace {
constexpr int kMaxDevices = 64;
std::atomic<int> g_sms[kMaxDevices];
std::atomic<int> g_smem[kMaxDevices];

int cached_attr(std::atomic<int>* table, cudaDeviceAttr attr, int fallback) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return fallback;
    int v = table[dev].load(std::memory_order_relaxed);
    if (v > 0) return v;
    if (cudaDeviceGetAttribute(&v, attr, dev) != cudaSuccess || v <= 0) return fallback;
    table[dev].store(v, std::memory_order_relaxed);
    return v;
}
}  // namespace

int num_sms() { return cached_attr(g_sms, cudaDevAttrMultiProcessorCount, 148); }

int max_smem_optin() {
    return cached_attr(g_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, 227 * 1024);
}

}  // namespace sd

extern "C" int sd_version(void) { return 100; }

extern "C" const char* sd_status_string(sd_status s) {
    switch (s) {
        case SD_OK: return "ok";
        case SD_ERR_INVALID_ARG: return "invalid argument";
        case SD_ERR_UNSUPPORTED: return "unsupported configuration";
        case SD_ERR_CUDA: return "CUDA error";
        case SD_ERR_DEVICE_BOUNDS: return "device-side bounds error";
        case SD_ERR_TIMEOUT: return "device-side wait timed out";
    }
    return "unknown status";
}

extern "C" const char* sd_last_error_message(void) { return sd::g_err; }
