// attend_noalloc.cu -- sd_gather_attend_noalloc: the gather-attend call for callers that
// cannot allocate device memory.
//
// sd_gather_attend needs a scratch buffer for its split-K partials, which the caller
// normally allocates once.  Some callers cannot do that: a plugin handed only raw input and
// output pointers by a host framework that owns all device memory, an engine that plans
// its whole memory budget at start-up and forbids allocations afterwards, or a plain C
// caller with no allocator at hand (cudaMalloc may also synchronize the device, which a
// latency-sensitive loop cannot afford).  For them this entry point takes the scratch from
// a fixed array compiled into the library instead.
//
// The array is kNoAllocScratchBytes (16 MiB) of device memory that every GPU which loads
// the library holds until the process exits.  On the first call made while a device is
// current, its device address is looked up with cudaGetSymbolAddress and the array is
// cleared once with cudaMemset (so make that first call before any stream capture).  The
// address is kept for the life of the process: after cudaDeviceReset it would be stale, so
// the call must not be used on a device that was reset.  All
// calls share the one array and it keeps whatever the last call left there.  The split
// partials are rewritten by every call before they are read, so nothing in the array needs
// to start at zero.
// Two calls whose kernels overlap on the GPU (different streams, no ordering between
// them) race on the array and give wrong results.  Requests whose split-K scratch needs
// more than the array holds are rejected with SD_ERR_INVALID_ARG before anything is
// launched.
#include <cuda_runtime.h>

#include <mutex>

#include "sd_host.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_attend_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices];

// Device address of g_attend_scratch on the current device (looked up once per device).
sd_status scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        sd::set_error("sd_gather_attend_noalloc: cudaGetDevice: %s", cudaGetErrorString(e));
        return SD_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) {
        sd::set_error("sd_gather_attend_noalloc: device ordinal %d out of range", dev);
        return SD_ERR_UNSUPPORTED;
    }
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_attend_scratch);
        if (e != cudaSuccess || p == nullptr) {
            sd::set_error("sd_gather_attend_noalloc: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
            return SD_ERR_CUDA;
        }
        e = cudaMemset(p, 0, kNoAllocScratchBytes);  // a defined start (nothing needs it)
        if (e != cudaSuccess) {
            sd::set_error("sd_gather_attend_noalloc: clearing the scratch: %s", cudaGetErrorString(e));
            return SD_ERR_CUDA;
        }
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return SD_OK;
}

}  // namespace

extern "C" sd_status sd_gather_attend_noalloc(const sd_attend_args* args, void* stream) {
    sd::clear_error();
    if (args == nullptr) {
        sd::set_error("sd_gather_attend_noalloc: null args");
        return SD_ERR_INVALID_ARG;
    }
    // Same split plan as sd_gather_attend; an invalid request reports its error there.
    const size_t need = sd_gather_attend_workspace_bytes(args);
    if (need > kNoAllocScratchBytes) {
        sd::set_error(
            "sd_gather_attend_noalloc: this request needs %zu bytes of split-K scratch, more than "
            "the %zu-byte static scratch; use sd_gather_attend with a workspace, or fewer splits",
            need, kNoAllocScratchBytes);
        return SD_ERR_INVALID_ARG;
    }
    void* scratch = nullptr;
    if (need > 0) {
        sd_status s = scratch_address(&scratch);
        if (s != SD_OK) return s;
    }
    sd_attend_args a = *args;
    a.workspace = scratch;
    a.workspace_bytes = need > 0 ? kNoAllocScratchBytes : 0;
    return sd_gather_attend(&a, stream);
}
