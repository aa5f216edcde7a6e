// gdn_prefill_noalloc: the prefill for callers that cannot allocate device
// memory.  A prefill with the short convolution needs a scratch buffer for the
// convolution's output; gdn_prefill_ex takes it from the caller.  Some callers
// have no way to provide one: a serving runtime that has handed all device
// memory to its own pool and may not call cudaMalloc on the request path, or
// code that must not allocate because an allocation can synchronise the
// device and break a latency budget.  This entry point uses a fixed scratch
// array that is part of the library itself instead.
//
// The array is a file-scope __device__ variable of kNoAllocScratchBytes.  With
// the CUDA runtime's default lazy module loading, its device memory is
// reserved when this file's module is first loaded on a device, which the
// first call on that device does (cudaGetSymbolAddress, made once per device
// with that device current, loads the module and returns the address); it then
// stays reserved until the process exits.  That first call should therefore
// come at initialisation: before the caller's own pool takes the device's
// memory (else the lookup fails for lack of memory and the call returns
// GDN_ERR_CUDA) and before any stream capture.  Later calls on that device
// allocate nothing.  All calls share the one array: calls whose work overlaps
// on the GPU (different streams, or several host threads) race on it and
// must be serialised by the caller.  Nothing in the array has to start at
// zero: every kernel writes each scratch element it reads (the convolution's
// output, the chunk records, the segment maps) before reading it.
#include <mutex>

#include "gdn_common.cuh"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;   // 32 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once).
cudaError_t scratch_for_current_device(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (g_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" {

size_t gdn_noalloc_scratch_bytes(void) { return kNoAllocScratchBytes; }

int gdn_prefill_noalloc(const gdn_prefill_desc* d, gdn_stream_t stream) {
    if (d == nullptr) return GDN_ERR_INVALID_ARG;
    if (gdn_workspace_bytes(d) == size_t(-1)) return gdn_prefill_ex(d, stream);   // let it report the error
    // Only the convolution's output must fit; the chunk records and the
    // segment maps are used when they fit as well (gdn_prefill_ex takes the
    // faster plans only when the workspace holds them).
    if (gdn::prefill_required_workspace(d) > kNoAllocScratchBytes) return GDN_ERR_TOO_LARGE;
    void* scratch = nullptr;
    const cudaError_t e = scratch_for_current_device(&scratch);
    if (e != cudaSuccess) return GDN_ERR_CUDA;
    gdn_prefill_desc local = *d;
    local.workspace = scratch;
    local.workspace_bytes = kNoAllocScratchBytes;
    return gdn_prefill_ex(&local, stream);
}

}  // extern "C"
