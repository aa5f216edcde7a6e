// Short-convolution prologue: the depthwise causal convolution over the
// previous conv state plus the prompt's columns, and the new conv state (the
// last K-1 columns), as add_short_conv_rows does ("perf(mamba): prefill text
// prompts in multi-token chunks", Implementation; reused by the Qwen3.5 page's
// Implementation section).
//
// For channel c of sequence n, xx = [state_in[n, c, 0..K-2], x[cu[n].., c]]
// (oldest first) and y_t = act(sum_{j<K} w[c, j] xx[t + j]); tap K-1 weighs
// the current token.  HBM-bound: each thread produces one (token, channel)
// output; consecutive threads take consecutive channels so that every load
// and store of a warp is one contiguous segment.
#include "gdn_common.cuh"

namespace gdn {
namespace {

constexpr int kConvThreads = 256;
constexpr int kConvTokensPerBlock = 8;

__device__ __forceinline__ float act_fn(float y, int act) {
    return act == GDN_ACT_SILU ? y / (1.f + expf(-y)) : y;
}

// Sequence holding token t: the n with cu[n] <= t < cu[n+1] (binary search;
// empty sequences are skipped because their range is empty).
__device__ __forceinline__ int find_seq(const int32_t* cu, int B, int64_t t) {
    int lo = 0, hi = B - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (int64_t(cu[mid]) <= t) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

template <typename Tin>
__global__ void __launch_bounds__(kConvThreads) conv_kernel(const ConvParams p) {
    const int c = blockIdx.y * kConvThreads + threadIdx.x;
    if (c >= p.C) return;
    const Tin* x = static_cast<const Tin*>(p.x);
    Tin* y = static_cast<Tin*>(p.y);
    const int K = p.K;
    float w[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) w[j] = j < K ? p.w[int64_t(c) * K + j] : 0.f;
    const int64_t tb = int64_t(blockIdx.x) * kConvTokensPerBlock;
    for (int r = 0; r < kConvTokensPerBlock; ++r) {
        const int64_t t = tb + r;
        if (t >= p.T) return;
        const int n = find_seq(p.cu, p.B, t);
        int64_t start = p.cu[n];
        if (start > t) start = t;   // only with a malformed cu_seqlens: stay in bounds
        float acc = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if (j < K) {
                const int64_t tt = t - (K - 1) + j;
                float xv;
                if (tt >= start) {
                    xv = load_elem(x, tt * p.C + c);
                } else {
                    const int64_t si = tt - start + (K - 1);   // index into the K-1 state columns
                    xv = p.state_in ? p.state_in[(int64_t(n) * p.C + c) * (K - 1) + si] : 0.f;
                }
                acc = fmaf(w[j], xv, acc);
            }
        }
        store_elem(y, t * p.C + c, act_fn(acc, p.act));
    }
}

// New conv state: the last K-1 entries of xx.  Reads every input column
// before writing, so state_out may alias state_in.  Runs after conv_kernel on
// the same stream, so no reader of the old state is still in flight.
template <typename Tin>
__global__ void __launch_bounds__(kConvThreads) conv_state_kernel(const ConvParams p) {
    const int64_t idx = int64_t(blockIdx.x) * kConvThreads + threadIdx.x;
    if (idx >= int64_t(p.B) * p.C) return;
    const int n = int(idx / p.C), c = int(idx % p.C);
    const int K = p.K;
    const Tin* x = static_cast<const Tin*>(p.x);
    const int64_t start = p.cu[n];
    int64_t L = int64_t(p.cu[n + 1]) - start;
    if (L < 0) L = 0;               // only with a malformed cu_seqlens: stay in bounds
    float keep[7];
#pragma unroll
    for (int j = 0; j < 7; ++j) {
        if (j < K - 1) {
            const int64_t xi = L + j;               // index into xx (length L + K - 1)
            if (xi < K - 1)
                keep[j] = p.state_in ? p.state_in[idx * (K - 1) + xi] : 0.f;
            else
                keep[j] = load_elem(x, (start + xi - (K - 1)) * p.C + c);
        }
    }
#pragma unroll
    for (int j = 0; j < 7; ++j)
        if (j < K - 1) p.state_out[idx * (K - 1) + j] = keep[j];
}

}  // namespace

cudaError_t launch_conv(const ConvParams& p, int dtype, cudaStream_t s) {
    if (p.T == 0) return cudaSuccess;
    const dim3 grid(unsigned((p.T + kConvTokensPerBlock - 1) / kConvTokensPerBlock),
                    (p.C + kConvThreads - 1) / kConvThreads);
    timer_begin(s, "conv_kernel");
    if (dtype == GDN_FP32)
        conv_kernel<float><<<grid, kConvThreads, 0, s>>>(p);
    else
        conv_kernel<__nv_bfloat16><<<grid, kConvThreads, 0, s>>>(p);
    timer_end(s);
    return cudaGetLastError();
}

cudaError_t launch_conv_state(const ConvParams& p, int dtype, cudaStream_t s) {
    const int64_t n = int64_t(p.B) * p.C;
    if (n == 0 || p.state_out == nullptr) return cudaSuccess;
    const unsigned blocks = unsigned((n + kConvThreads - 1) / kConvThreads);
    timer_begin(s, "conv_state_kernel");
    if (dtype == GDN_FP32)
        conv_state_kernel<float><<<blocks, kConvThreads, 0, s>>>(p);
    else
        conv_state_kernel<__nv_bfloat16><<<blocks, kConvThreads, 0, s>>>(p);
    timer_end(s);
    return cudaGetLastError();
}

}  // namespace gdn
