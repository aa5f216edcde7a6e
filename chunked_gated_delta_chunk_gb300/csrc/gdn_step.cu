// One-token decode step of the gated delta rule (the unchanged one-token
// decoder step of "perf(qwen3_5): prefill text prompts in multi-token
// chunks", Exit Criteria: decode stays on the one-token engine), reading and
// writing the same recurrent-state layout as the prefill:
//
//   S <- exp(g) S;  u = beta (v - S^T k);  S <- S + k u^T;  o = q_scale S^T q
//
// with the optional short-convolution step in front (one new column per
// sequence) and the q/k L2 normalisation.  HBM-bound over the fp32 state:
// grid (dv / NS slabs, Hv, B); a CTA streams its [dk, NS] state slab once in
// and once out, each warp reading 32 consecutive floats of a state row.
#include "gdn_common.cuh"

namespace gdn {
namespace {

constexpr int kStepThreads = 128;
constexpr int kMaxRowsPerThread = 32;   // dk / (128 / NS) with dk <= 128, NS = 32

__device__ __forceinline__ float act_fn(float y, int act) {
    return act == GDN_ACT_SILU ? y / (1.f + expf(-y)) : y;
}

// Input channel value for the current token: the raw tensor, or the short
// convolution over [conv state, the token's column].
template <typename Tin>
__device__ __forceinline__ float step_input(const StepParams& p, const Tin* plain, int64_t plain_idx,
                                            int n, int c) {
    if (p.conv_x == nullptr) return load_elem(plain, plain_idx);
    const int C = 2 * p.Hk * p.dk + p.Hv * p.dv;
    const int K = p.conv_K;
    const float* w = p.conv_w + int64_t(c) * K;
    float acc = w[K - 1] * load_elem(static_cast<const Tin*>(p.conv_x), int64_t(n) * C + c);
    if (p.conv_state_in) {
        const float* st = p.conv_state_in + (int64_t(n) * C + c) * (K - 1);
        for (int j = 0; j < K - 1; ++j) acc = fmaf(w[j], st[j], acc);
    }
    return act_fn(acc, p.conv_act);
}

template <typename Tin>
__global__ void __launch_bounds__(kStepThreads) step_kernel(const StepParams p) {
    const int slab = blockIdx.x, h = blockIdx.y, n = blockIdx.z;
    const int dk = p.dk, dv = p.dv;
    const int NS = dv < 32 ? dv : 32;
    const int RG = kStepThreads / NS;                // row groups
    const int j0 = slab * NS;
    const int kh = h / (p.Hv / p.Hk);
    const int tid = threadIdx.x;
    const int jj = tid % NS, rg = tid / NS;
    const int warp = tid >> 5, lane = tid & 31;

    __shared__ float sq[128], sk[128], sv[32];
    __shared__ float sred[kStepThreads];
    __shared__ float su[32];

    const Tin* q = static_cast<const Tin*>(p.q);
    const Tin* k = static_cast<const Tin*>(p.k);
    const Tin* v = static_cast<const Tin*>(p.v);
    const int qoff = kh * dk, koff = p.Hk * dk + kh * dk, voff = 2 * p.Hk * dk + h * dv;
    for (int d = tid; d < dk; d += kStepThreads) {
        sq[d] = step_input(p, q, (int64_t(n) * p.Hk + kh) * dk + d, n, qoff + d);
        sk[d] = step_input(p, k, (int64_t(n) * p.Hk + kh) * dk + d, n, koff + d);
    }
    for (int j = tid; j < NS; j += kStepThreads)
        sv[j] = step_input(p, v, (int64_t(n) * p.Hv + h) * dv + j0 + j, n, voff + j0 + j);
    __syncthreads();
    if (p.l2norm && warp < 2) {
        float* row = warp == 0 ? sq : sk;
        float ss = 0.f;
        for (int d = lane; d < dk; d += 32) ss = fmaf(row[d], row[d], ss);
        ss = warp_sum(ss);
        const float inv = rsqrtf(ss + p.eps);
        for (int d = lane; d < dk; d += 32) row[d] *= inv;
    }
    __syncthreads();

    const float decay = expf(p.g[int64_t(n) * p.Hv + h]);
    const float b = p.beta[int64_t(n) * p.Hv + h];
    const size_t sbase = (size_t(n) * p.Hv + h) * size_t(dk) * dv + j0 + jj;
    float s[kMaxRowsPerThread];
    float kv = 0.f;
#pragma unroll
    for (int r = 0; r < kMaxRowsPerThread; ++r) {
        const int i = rg + r * RG;
        if (i < dk) {
            const float x = p.state_in ? p.state_in[sbase + size_t(i) * dv] * decay : 0.f;
            s[r] = x;
            kv = fmaf(x, sk[i], kv);
        }
    }
    sred[tid] = kv;
    __syncthreads();
    if (tid < NS) {
        float acc = 0.f;
        for (int g2 = 0; g2 < RG; ++g2) acc += sred[g2 * NS + tid];
        su[tid] = b * (sv[tid] - acc);
    }
    __syncthreads();
    const float u = su[jj];
    float o = 0.f;
#pragma unroll
    for (int r = 0; r < kMaxRowsPerThread; ++r) {
        const int i = rg + r * RG;
        if (i < dk) {
            const float x = fmaf(sk[i], u, s[r]);
            o = fmaf(x, sq[i], o);
            if (p.state_out) p.state_out[sbase + size_t(i) * dv] = x;
        }
    }
    __syncthreads();
    sred[tid] = o;
    __syncthreads();
    if (tid < NS) {
        float acc = 0.f;
        for (int g2 = 0; g2 < RG; ++g2) acc += sred[g2 * NS + tid];
        store_elem(static_cast<Tin*>(p.out), (int64_t(n) * p.Hv + h) * dv + j0 + tid,
                   acc * p.q_scale);
    }
}

// conv_state_out[n, c, :] = [conv_state_in[n, c, 1:], x[n, c]]: launched after
// step_kernel on the same stream, so every reader of the old state is done;
// each thread reads its whole row before writing, so the two may alias.
template <typename Tin>
__global__ void __launch_bounds__(256) step_conv_state_kernel(const StepParams p) {
    const int C = 2 * p.Hk * p.dk + p.Hv * p.dv;
    const int64_t idx = int64_t(blockIdx.x) * 256 + threadIdx.x;
    if (idx >= int64_t(p.B) * C) return;
    const int K = p.conv_K;
    float keep[7];
#pragma unroll
    for (int j = 0; j < 7; ++j) {
        if (j < K - 1) {
            if (j + 1 < K - 1)
                keep[j] = p.conv_state_in ? p.conv_state_in[idx * (K - 1) + j + 1] : 0.f;
            else
                keep[j] = load_elem(static_cast<const Tin*>(p.conv_x), idx);
        }
    }
#pragma unroll
    for (int j = 0; j < 7; ++j)
        if (j < K - 1) p.conv_state_out[idx * (K - 1) + j] = keep[j];
}

}  // namespace

cudaError_t launch_step(const StepParams& p, int dtype, cudaStream_t s) {
    if (p.B == 0) return cudaSuccess;
    const int NS = p.dv < 32 ? p.dv : 32;
    const dim3 grid(p.dv / NS, p.Hv, p.B);
    timer_begin(s, "step_kernel");
    if (dtype == GDN_FP32)
        step_kernel<float><<<grid, kStepThreads, 0, s>>>(p);
    else
        step_kernel<__nv_bfloat16><<<grid, kStepThreads, 0, s>>>(p);
    timer_end(s);
    return cudaGetLastError();
}

cudaError_t launch_step_conv_state(const StepParams& p, int dtype, cudaStream_t s) {
    const int C = 2 * p.Hk * p.dk + p.Hv * p.dv;
    const int64_t n = int64_t(p.B) * C;
    if (n == 0 || p.conv_x == nullptr || p.conv_state_out == nullptr) return cudaSuccess;
    const unsigned blocks = unsigned((n + 255) / 256);
    timer_begin(s, "step_conv_state_kernel");
    if (dtype == GDN_FP32)
        step_conv_state_kernel<float><<<blocks, 256, 0, s>>>(p);
    else
        step_conv_state_kernel<__nv_bfloat16><<<blocks, 256, 0, s>>>(p);
    timer_end(s);
    return cudaGetLastError();
}

}  // namespace gdn
