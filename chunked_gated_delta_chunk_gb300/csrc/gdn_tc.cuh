// Tensor-core (tcgen05) chunk path: declarations used by the C ABI layer.
#pragma once

#include "gdn_common.cuh"

namespace gdn {

constexpr const char* kTcKernelName = "chunk_tc_kernel";

// True when the tensor-core kernel handles this call: bf16 with dk = dv = 128.
inline bool tc_supported(const ChunkParams& p, int dtype) {
    return dtype == GDN_BF16 && p.dk == 128 && p.dv == 128;
}

// Encodes the TMA maps and launches one CTA per (value head, sequence).
cudaError_t launch_chunk_tc(const ChunkParams& p, cudaStream_t s);

}  // namespace gdn
