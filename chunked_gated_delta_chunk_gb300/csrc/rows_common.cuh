// Device helpers shared by the row-recurrence kernels (selective-scan rows,
// RWKV-4 WKV rows): the ticket/flag protocol of their decoupled look-back and
// the sequence lookup in cu_seqlens.
#pragma once

#include <stdint.h>

#include "tc_ptx.cuh"

namespace gdn {
namespace rows {

constexpr int kScanRows = 64;          // rows of a selective-scan tile (a, b: 16 KB, many CTAs per SM)
constexpr int kWkvRows = 128;          // rows of a WKV tile (k, v: 32 KB; the WKV rows carry more arithmetic)
constexpr int kCols = 32;              // channels of a tile (one lane each)
constexpr int kWarps = 4;              // warp w owns rows 64 w .. 64 w + 63
constexpr int kThreads = 32 * kWarps;
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

constexpr int kChains = 4;             // independent row chains per thread
enum : int { kRowStart = 1, kRowEnd = 2 };

// Sequence and start / end marks of the tile's rows (all threads of the CTA
// share the rows); the caller synchronises before reading them.
__device__ __forceinline__ void fill_row_info(const int32_t* cu, int B, int64_t t0, int nrow, int tid,
                                              int* seq, int* mark) {
    for (int r = tid; r < nrow; r += kThreads) {
        const int64_t t = t0 + r;
        const int n = find_seq(cu, B, t);
        seq[r] = n;
        mark[r] = (t == cu[n] ? kRowStart : 0) | (t == int64_t(cu[n + 1]) - 1 ? kRowEnd : 0);
    }
}

// Stage rows [t0, t0 + nrow) x channels [c0, c0 + kCols) of two [T, C] fp32
// arrays into [kRows][kCols] shared tiles by 16-byte cp.async (C a multiple
// of 4); rows and channels outside are zero.
template <int R>
__device__ __forceinline__ void stage_tile(float* sx, float* sy, const float* x, const float* y,
                                           int64_t t0, int nrow, int c0, int C, int tid) {
    for (int i = tid; i < R * (kCols / 4); i += kThreads) {
        const int r = i / (kCols / 4), q = (i % (kCols / 4)) * 4;
        float* dx = sx + r * kCols + q;
        float* dy = sy + r * kCols + q;
        if (r < nrow && c0 + q < C) {
            const int64_t off = (t0 + r) * C + c0 + q;
            ptx::cp_async16(dx, x + off);
            ptx::cp_async16(dy, y + off);
        } else {
            *reinterpret_cast<float4*>(dx) = make_float4(0.f, 0.f, 0.f, 0.f);
            *reinterpret_cast<float4*>(dy) = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    ptx::cp_async_commit();
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
