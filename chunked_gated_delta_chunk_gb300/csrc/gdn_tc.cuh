// Tensor-core (tcgen05) chunk path: declarations used by the C ABI layer.
#pragma once

#include "gdn_common.cuh"

namespace gdn {

constexpr const char* kTcKernelName = "chunk_tc_kernel";

// True when the tensor-core kernel handles this call (bf16, dk = dv = 128).
inline bool tc_supported(const ChunkParams& p, int dtype) {
    (void)p;
    (void)dtype;
    return false;
}

inline cudaError_t launch_chunk_tc(const ChunkParams& p, cudaStream_t s) {
    (void)p;
    (void)s;
    return cudaErrorNotSupported;
}

}  // namespace gdn
