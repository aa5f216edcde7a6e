// Short-convolution prologue: the depthwise causal convolution over the
// previous conv state plus the prompt's columns, and the new conv state (the
// last K-1 columns), as add_short_conv_rows does ("perf(mamba): prefill text
// prompts in multi-token chunks", Implementation; reused by the Qwen3.5 page's
// Implementation section).
//
// For channel c of sequence n, xx = [state_in[n, c, 0..K-2], x[cu[n].., c]]
// (oldest first) and y_t = act(sum_{j<K} w[c, j] xx[t + j]); tap K-1 weighs
// the current token.  HBM-bound: consecutive threads take consecutive groups
// of 8 channels, so every 16-byte load and store of a warp is one contiguous
// 512-byte segment of a token row.
#include "gdn_common.cuh"
#include "tc_ptx.cuh"

namespace gdn {
namespace {

constexpr int kConvThreads = 128;
constexpr int kConvRun = 128;           // tokens per thread (fewer halo re-reads)
constexpr int kConvGroup = 8;           // token rows loaded together

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

// 8 consecutive channels of one token row as floats (16-byte aligned: C is a
// multiple of 16 and the row base is 16-byte aligned).
__device__ __forceinline__ void load8(const __nv_bfloat16* p, float* v) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(b[i]);
        v[2 * i] = f.x;
        v[2 * i + 1] = f.y;
    }
}
__device__ __forceinline__ void load8(const float* p, float* v) {
    const float4 a = *reinterpret_cast<const float4*>(p), b = *reinterpret_cast<const float4*>(p + 4);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
// Raw 16-byte words of 8 channels, kept packed while a group of rows is in
// flight (bf16: one word, fp32: two), unpacked to floats when used.
template <typename Tin> struct Raw8;
template <> struct Raw8<__nv_bfloat16> {
    uint4 w;
    __device__ __forceinline__ void load(const __nv_bfloat16* p) { w = *reinterpret_cast<const uint4*>(p); }
    __device__ __forceinline__ void unpack(float* v) const {
        const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __bfloat1622float2(b[i]);
            v[2 * i] = f.x;
            v[2 * i + 1] = f.y;
        }
    }
};
template <> struct Raw8<float> {
    float4 a, b;
    __device__ __forceinline__ void load(const float* p) {
        a = *reinterpret_cast<const float4*>(p);
        b = *reinterpret_cast<const float4*>(p + 4);
    }
    __device__ __forceinline__ void unpack(float* v) const {
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    }
};

__device__ __forceinline__ void store8(__nv_bfloat16* p, const float* v) {
    uint4 u;
    uint32_t* w = reinterpret_cast<uint32_t*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __nv_bfloat162 b = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
        w[i] = *reinterpret_cast<const uint32_t*>(&b);
    }
    *reinterpret_cast<uint4*>(p) = u;
}
__device__ __forceinline__ void store8(float* p, const float* v) {
    *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
    *reinterpret_cast<float4*>(p + 4) = make_float4(v[4], v[5], v[6], v[7]);
}

// One thread: 8 consecutive channels over a run of kConvRun tokens.  The K-1
// previous columns of xx stay in registers as a sliding window, so every
// input row is read once; a sequence start inside the run reloads the window
// from that sequence's conv state.
template <typename Tin, int K>
__global__ void __launch_bounds__(kConvThreads) conv_kernel(const ConvParams p) {
    ptx::griddep_wait();                      // the grid before may still read the workspace
    const int c0 = (blockIdx.y * kConvThreads + threadIdx.x) * 8;
    if (c0 >= p.C) return;
    const int64_t t0 = int64_t(blockIdx.x) * kConvRun;
    if (t0 >= p.T) return;
    const int64_t t1 = t0 + kConvRun < p.T ? t0 + kConvRun : p.T;
    const Tin* x = static_cast<const Tin*>(p.x);
    Tin* y = static_cast<Tin*>(p.y);
    float w[8][K];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < K; ++j) w[i][j] = p.w[int64_t(c0 + i) * K + j];
    float win[K - 1][8];        // win[j] = xx column t - (K - 1) + j
    int n = find_seq(p.cu, p.B, t0);
    int64_t start = p.cu[n], stop = p.cu[n + 1];
    // columns t - K + 1 .. t - 1 of sequence n: inputs at or after its start,
    // else its conv state (oldest first), else zero
    auto fill_window = [&](int64_t t) {
#pragma unroll
        for (int j = 0; j < K - 1; ++j) {
            const int64_t tt = t - (K - 1) + j;
            if (tt >= start) {
                load8(x + tt * p.C + c0, win[j]);
            } else {
                const int64_t si = tt - start + (K - 1);
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    win[j][i] = (p.state_in && si >= 0) ? p.state_in[(int64_t(n) * p.C + c0 + i) * (K - 1) + si] : 0.f;
            }
        }
    };
    if (start > t0) start = t0;   // only with a malformed cu_seqlens: stay in bounds
    fill_window(t0);
    // one output column from the window and the current input; then slide
    auto emit = [&](int64_t t, const float* cur) {
        float out[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            float acc = 0.f;
#pragma unroll
            for (int j = 0; j < K - 1; ++j) acc = fmaf(w[i][j], win[j][i], acc);
            acc = fmaf(w[i][K - 1], cur[i], acc);
            out[i] = act_fn(acc, p.act);
        }
        store8(y + t * p.C + c0, out);
#pragma unroll
        for (int j = 0; j + 1 < K - 1; ++j)
#pragma unroll
            for (int i = 0; i < 8; ++i) win[j][i] = win[j + 1][i];
#pragma unroll
        for (int i = 0; i < 8; ++i) win[K - 2][i] = cur[i];
    };
    for (int64_t t = t0; t < t1;) {
        if (t >= stop) {                            // next non-empty sequence starts here
            while (n + 1 < p.B && int64_t(p.cu[n + 1]) <= t) ++n;
            start = p.cu[n];
            stop = p.cu[n + 1];
            if (start > t) start = t;
            if (stop <= t) stop = p.T;              // malformed cu_seqlens: stay in bounds
            fill_window(t);
        }
        const int64_t end = t1 < stop ? t1 : stop;  // tokens of this sequence in the run
        // groups of kConvGroup rows: all loads of a group in flight together
        for (; t + kConvGroup <= end; t += kConvGroup) {
            Raw8<Tin> raw[kConvGroup];
#pragma unroll
            for (int u = 0; u < kConvGroup; ++u) raw[u].load(x + (t + u) * p.C + c0);
#pragma unroll
            for (int u = 0; u < kConvGroup; ++u) {
                float cur[8];
                raw[u].unpack(cur);
                emit(t + u, cur);
            }
        }
        for (; t < end; ++t) {
            float cur[8];
            load8(x + t * p.C + c0, cur);
            emit(t, cur);
        }
    }
}

// New conv state: the last K-1 entries of xx.  Reads every input column
// before writing, so state_out may alias state_in.  Runs after conv_kernel on
// the same stream, so no reader of the old state is still in flight.
template <typename Tin>
__global__ void __launch_bounds__(kConvThreads) conv_state_kernel(const ConvParams p) {
    ptx::griddep_wait();                      // the conv state is read and written in place
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

template <typename Tin>
cudaError_t launch_conv_k(const ConvParams& p, dim3 grid, cudaStream_t s) {
    switch (p.K) {
        case 2: return launch_pdl(conv_kernel<Tin, 2>, grid, kConvThreads, 0, s, p);
        case 3: return launch_pdl(conv_kernel<Tin, 3>, grid, kConvThreads, 0, s, p);
        case 4: return launch_pdl(conv_kernel<Tin, 4>, grid, kConvThreads, 0, s, p);
        case 5: return launch_pdl(conv_kernel<Tin, 5>, grid, kConvThreads, 0, s, p);
        case 6: return launch_pdl(conv_kernel<Tin, 6>, grid, kConvThreads, 0, s, p);
        case 7: return launch_pdl(conv_kernel<Tin, 7>, grid, kConvThreads, 0, s, p);
        default: return launch_pdl(conv_kernel<Tin, 8>, grid, kConvThreads, 0, s, p);
    }
}

}  // namespace

cudaError_t launch_conv(const ConvParams& p, int dtype, cudaStream_t s) {
    if (p.T == 0) return cudaSuccess;
    const dim3 grid(unsigned((p.T + kConvRun - 1) / kConvRun),
                    (p.C / 8 + kConvThreads - 1) / kConvThreads);
    timer_begin(s, "conv_kernel");
    const cudaError_t e = dtype == GDN_FP32 ? launch_conv_k<float>(p, grid, s) : launch_conv_k<__nv_bfloat16>(p, grid, s);
    timer_end(s);
    return e;
}

cudaError_t launch_conv_state(const ConvParams& p, int dtype, cudaStream_t s) {
    const int64_t n = int64_t(p.B) * p.C;
    if (n == 0 || p.state_out == nullptr) return cudaSuccess;
    const unsigned blocks = unsigned((n + kConvThreads - 1) / kConvThreads);
    timer_begin(s, "conv_state_kernel");
    const cudaError_t e = dtype == GDN_FP32
                              ? launch_pdl(conv_state_kernel<float>, dim3(blocks), kConvThreads, 0, s, p)
                              : launch_pdl(conv_state_kernel<__nv_bfloat16>, dim3(blocks), kConvThreads, 0, s, p);
    timer_end(s);
    return e;
}

}  // namespace gdn
