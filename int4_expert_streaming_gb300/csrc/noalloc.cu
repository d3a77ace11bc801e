// noalloc.cu -- fixed device scratch for moe_route_noalloc: the routing of a
// decode batch with no allocation inside the call.
//
// The array lives in this translation unit; its device address is looked up
// once per device with cudaGetSymbolAddress (the first call on a device does
// that lookup, so it should come before any stream capture) and cached.
#include <cuda_runtime.h>

#include <mutex>

namespace moe {

constexpr size_t kNoallocScratchBytes = 256 * 1024;  // modest fixed size: 256 KiB

static __device__ __align__(256) unsigned char g_route_scratch[kNoallocScratchBytes];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices] = {};
}  // namespace

// Device address of the scratch array on `device` (the current device).
// Returns cudaSuccess and the address, or the lookup's error.
cudaError_t noalloc_scratch(int device, void** ptr, size_t* bytes) {
    *bytes = kNoallocScratchBytes;
    if (device < 0 || device >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_addr[device]) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_route_scratch);
        if (e != cudaSuccess) return e;
        g_addr[device] = p;
    }
    *ptr = g_addr[device];
    return cudaSuccess;
}

}  // namespace moe
