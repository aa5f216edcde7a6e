// Device helpers shared by the row-recurrence kernels (selective-scan rows,
// RWKV-4 WKV rows): the ticket/flag protocol of their decoupled look-back and
// the sequence lookup in cu_seqlens.
#pragma once

#include <stdint.h>

namespace gdn {
namespace rows {

constexpr int kRows = 64;              // rows of a tile
constexpr int kCols = 128;             // channels of a tile (one thread each)
constexpr uint32_t kSpinLimit = 1u << 22;

__device__ __forceinline__ int ld_acquire(const int* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release(int* p, int v) {
    asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Sequence holding row t: the largest n with cu[n] <= t (empty sequences
// before t are skipped).
__device__ __forceinline__ int find_seq(const int32_t* cu, int B, int64_t t) {
    int lo = 0, hi = B - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (int64_t(cu[mid]) <= t) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

// Thread 0 waits (bounded) until the tile flag is non-zero; returns it, or 0
// when the wait ran out.
__device__ __forceinline__ int wait_flag(const int* flag) {
    int f = 0;
    uint32_t it = 0;
    while ((f = ld_acquire(flag)) == 0 && ++it < kSpinLimit) __nanosleep(64);
    return f;
}

}  // namespace rows
}  // namespace gdn
