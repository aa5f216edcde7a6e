// SIMT fp32 chunk kernel: the closed-form chunk solve of "perf(qwen3_5):
// prefill text prompts in multi-token chunks" (Implementation section) in
// plain fp32 FMA arithmetic, with the state carried through the chunks of a
// sequence inside one CTA.
//
// This path serves the fp32 dtype (no TF32 anywhere, as the page's review of
// its 64-row solve asks for a full-FP32 check) and every supported head size
// (16, 32, 64, 128).  The tensor-core path handles bf16 with dk = dv = 128.
//
// Grid: (dv / NS value slabs, Hv, B); one CTA owns the state columns
// [j0, j0 + NS) of one (sequence, value head) and walks the sequence's chunks
// in order.  Columns of S evolve independently (every dk-side quantity is
// shared), so slabs need no communication.
//
// Per chunk of n <= 64 rows (gamma inclusive cumsum of g, Gamma = exp(gamma)):
//   A_ij = beta_i exp(gamma_i - gamma_j) k_i.k_j  (j < i)
//   T    = (I + A)^-1 on a 64-row identity padding: 8x8 diagonal blocks by
//          the Neumann product (I - N)(I + N^2)(I + N^4), then 2x2 block
//          inversion level by level (8 -> 16 -> 32 -> 64)
//   U    = T (diag(beta) V - diag(beta Gamma) K S_0)
//   O    = diag(Gamma) Q S_0 + (exp(gamma_t - gamma_i) q_t.k_i)_{i<=t} U
//   S_S  = exp(gamma_S) S_0 + (K * exp(min(gamma_S - gamma, 0)))^T U
// Exponentials are only evaluated where a triangular mask keeps the entry,
// and every exponent is clamped at zero (the page clamps gamma_S - gamma_i;
// for g <= 0 the other two are <= 0 already, the clamp only guards them).
#include <algorithm>

#include "gdn_common.cuh"

namespace gdn {
namespace {

constexpr int kThreads = 256;
constexpr int kLdA = kMaxChunk + 1;          // padded row stride of 64x64 tiles
constexpr int kTmpFloats = 8 * 3 * 64;        // per-warp N^2, N^4, X for 8 blocks

struct SmemLayout {
    int ldq, lds, ns;
    size_t q, k, v, s, a, t, p, ks, qs, u, tmp, gam, beta, eg, end, total;
};

__host__ __device__ inline SmemLayout smem_layout(int dk, int dv) {
    SmemLayout L;
    L.ns = dv < 32 ? dv : 32;
    L.ldq = dk + 1;
    L.lds = L.ns + 1;
    size_t o = 0;
    L.q = o;    o += size_t(kMaxChunk) * L.ldq;
    L.k = o;    o += size_t(kMaxChunk) * L.ldq;
    L.v = o;    o += size_t(kMaxChunk) * L.lds;
    L.s = o;    o += size_t(dk) * L.lds;
    L.a = o;    o += size_t(kMaxChunk) * kLdA;
    L.t = o;    o += size_t(kMaxChunk) * kLdA;
    L.p = o;    o += size_t(kMaxChunk) * kLdA;
    L.ks = o;   o += size_t(kMaxChunk) * L.lds;
    L.qs = o;   o += size_t(kMaxChunk) * L.lds;
    L.u = o;    o += size_t(kMaxChunk) * L.lds;
    L.tmp = o;  o += kTmpFloats;
    L.gam = o;  o += kMaxChunk;
    L.beta = o; o += kMaxChunk;
    L.eg = o;   o += kMaxChunk;
    L.end = o;  o += kMaxChunk;
    L.total = o * sizeof(float);
    return L;
}

// T = (I + A)^-1 for the strictly lower 64x64 A in sA (padded rows are zero,
// so T is identity there).  All threads of the CTA take part.
__device__ void block_inverse_64(const float* sA, float* sT, float* sTmp) {
    const int tid = threadIdx.x, nth = blockDim.x;
    const int warp = tid >> 5, lane = tid & 31;
    for (int idx = tid; idx < kMaxChunk * kLdA; idx += nth) sT[idx] = 0.f;
    __syncthreads();

    // Stage 1: warp w inverts diagonal block w (8 warps, 8 blocks).
    if (warp < kMaxChunk / kNeumann) {
        const int o = warp * kNeumann;
        float* N2 = sTmp + warp * 192;
        float* N4 = N2 + 64;
        float* X = N4 + 64;
        auto N = [&](int r, int c) { return sA[(o + r) * kLdA + o + c]; };
        for (int e = lane; e < 64; e += 32) {
            int r = e >> 3, c = e & 7;
            float acc = 0.f;
            for (int m = 0; m < 8; ++m) acc = fmaf(N(r, m), N(m, c), acc);
            N2[e] = acc;
        }
        __syncwarp();
        for (int e = lane; e < 64; e += 32) {
            int r = e >> 3, c = e & 7;
            float acc = 0.f, nn2 = 0.f;
            for (int m = 0; m < 8; ++m) {
                acc = fmaf(N2[r * 8 + m], N2[m * 8 + c], acc);
                nn2 = fmaf(N(r, m), N2[m * 8 + c], nn2);
            }
            N4[e] = acc;
            // X = (I - N)(I + N^2) = I - N + N^2 - N N^2
            X[e] = (r == c ? 1.f : 0.f) - N(r, c) + N2[e] - nn2;
        }
        __syncwarp();
        for (int e = lane; e < 64; e += 32) {
            int r = e >> 3, c = e & 7;
            float acc = X[e];                          // X (I + N^4)
            for (int m = 0; m < 8; ++m) acc = fmaf(X[r * 8 + m], N4[m * 8 + c], acc);
            sT[(o + r) * kLdA + o + c] = acc;
        }
    }
    __syncthreads();

    // Stage 2: [[L11, 0], [L21, L22]]^-1 has lower-left block -L22^-1 L21 L11^-1.
    for (int size = kNeumann; size < kMaxChunk; size *= 2) {
        const int pairs = kMaxChunk / (2 * size);
        const int per = size * size;
        for (int idx = tid; idx < pairs * per; idx += nth) {       // tmp = L21 L11^-1
            int pr = idx / per, r = (idx / size) % size, c = idx % size;
            int o = pr * 2 * size;
            float acc = 0.f;
            for (int m = c; m < size; ++m)
                acc = fmaf(sA[(o + size + r) * kLdA + o + m], sT[(o + m) * kLdA + o + c], acc);
            sTmp[idx] = acc;
        }
        __syncthreads();
        for (int idx = tid; idx < pairs * per; idx += nth) {       // -L22^-1 tmp
            int pr = idx / per, r = (idx / size) % size, c = idx % size;
            int o = pr * 2 * size;
            float acc = 0.f;
            for (int m = 0; m <= r; ++m)
                acc = fmaf(sT[(o + size + r) * kLdA + o + size + m], sTmp[pr * per + m * size + c], acc);
            sT[(o + size + r) * kLdA + o + c] = -acc;
        }
        __syncthreads();
    }
}

template <typename Tin>
__global__ void __launch_bounds__(kThreads) chunk_simt_kernel(const ChunkParams p) {
    const int slab = blockIdx.x, h = blockIdx.y, n = blockIdx.z;
    const int dk = p.dk, dv = p.dv;
    const SmemLayout L = smem_layout(dk, dv);
    const int NS = L.ns, ldq = L.ldq, lds = L.lds;
    const int j0 = slab * NS;
    const int kh = h / (p.Hv / p.Hk);
    const int tid = threadIdx.x, nth = blockDim.x;
    const int warp = tid >> 5, lane = tid & 31, nwarps = nth >> 5;

    extern __shared__ float smem[];
    float* sQ = smem + L.q;
    float* sK = smem + L.k;
    float* sV = smem + L.v;
    float* sS = smem + L.s;
    float* sA = smem + L.a;
    float* sT = smem + L.t;
    float* sP = smem + L.p;
    float* sKS = smem + L.ks;
    float* sQS = smem + L.qs;
    float* sU = smem + L.u;
    float* sTmp = smem + L.tmp;
    float* sGam = smem + L.gam;
    float* sBeta = smem + L.beta;
    float* sEg = smem + L.eg;
    float* sEnd = smem + L.end;

    const Tin* q = static_cast<const Tin*>(p.q);
    const Tin* k = static_cast<const Tin*>(p.k);
    const Tin* v = static_cast<const Tin*>(p.v);
    Tin* out = static_cast<Tin*>(p.out);

    int64_t t0 = p.cu[n], t1 = p.cu[n + 1];
    t0 = t0 < 0 ? 0 : (t0 > p.t_cap ? p.t_cap : t0);
    t1 = t1 < t0 ? t0 : (t1 > p.t_cap ? p.t_cap : t1);

    const size_t sbase = (size_t(n) * p.Hv + h) * size_t(dk) * dv + j0;
    for (int idx = tid; idx < dk * NS; idx += nth) {
        int i = idx / NS, j = idx % NS;
        sS[i * lds + j] = p.state_in ? p.state_in[sbase + size_t(i) * dv + j] : 0.f;
    }
    __syncthreads();

    for (int64_t c0 = t0; c0 < t1; c0 += p.chunk) {
        const int rows = int(t1 - c0 < p.chunk ? t1 - c0 : p.chunk);
        // ---- load the chunk ------------------------------------------------
        for (int idx = tid; idx < rows * dk; idx += nth) {
            int r = idx / dk, d = idx % dk;
            int64_t t = c0 + r;
            sQ[r * ldq + d] = load_elem(q, t * p.q_stride + int64_t(kh) * dk + d);
            sK[r * ldq + d] = load_elem(k, t * p.k_stride + int64_t(kh) * dk + d);
        }
        for (int idx = tid; idx < rows * NS; idx += nth) {
            int r = idx / NS, j = idx % NS;
            sV[r * lds + j] = load_elem(v, (c0 + r) * p.v_stride + int64_t(h) * dv + j0 + j);
        }
        if (tid < rows) {
            sGam[tid] = p.g[(c0 + tid) * p.Hv + h];
            sBeta[tid] = p.beta[(c0 + tid) * p.Hv + h];
        }
        __syncthreads();
        // ---- L2 norm of q and k rows; inclusive cumsum of g ------------------
        if (p.l2norm) {
            for (int task = warp; task < 2 * rows; task += nwarps) {
                float* row = task < rows ? sQ + task * ldq : sK + (task - rows) * ldq;
                float ss = 0.f;
                for (int d = lane; d < dk; d += 32) ss = fmaf(row[d], row[d], ss);
                ss = warp_sum(ss);
                const float inv = rsqrtf(ss + p.eps);
                for (int d = lane; d < dk; d += 32) row[d] *= inv;
            }
        }
        if (tid == 0) {
            float acc = 0.f;
            for (int r = 0; r < rows; ++r) {
                acc += sGam[r];
                sGam[r] = acc;
            }
        }
        __syncthreads();
        if (tid < rows) {
            const float gm = sGam[tid];
            sEg[tid] = expf(gm);
            sEnd[tid] = expf(fminf(sGam[rows - 1] - gm, 0.f));
        }
        // ---- A (strict lower) and the masked, decayed Q K^T (lower incl. diag)
        for (int idx = tid; idx < kMaxChunk * kMaxChunk; idx += nth) {
            const int i = idx >> 6, j = idx & 63;
            float a = 0.f, pq = 0.f;
            if (i < rows && j <= i) {
                float dkk = 0.f, dqk = 0.f;
                for (int d = 0; d < dk; ++d) {
                    const float kj = sK[j * ldq + d];
                    dkk = fmaf(sK[i * ldq + d], kj, dkk);
                    dqk = fmaf(sQ[i * ldq + d], kj, dqk);
                }
                const float e = expf(fminf(sGam[i] - sGam[j], 0.f));
                if (j < i) a = sBeta[i] * e * dkk;
                pq = e * dqk;
            }
            sA[i * kLdA + j] = a;
            sP[i * kLdA + j] = pq;
        }
        // ---- K S_0 and Q S_0 ---------------------------------------------------
        for (int idx = tid; idx < rows * NS; idx += nth) {
            const int i = idx / NS, j = idx % NS;
            float ks = 0.f, qs = 0.f;
            for (int d = 0; d < dk; ++d) {
                const float s = sS[d * lds + j];
                ks = fmaf(sK[i * ldq + d], s, ks);
                qs = fmaf(sQ[i * ldq + d], s, qs);
            }
            sKS[i * lds + j] = ks;
            sQS[i * lds + j] = qs;
        }
        __syncthreads();
        block_inverse_64(sA, sT, sTmp);
        // ---- right-hand side, in place: beta_i (v_i - Gamma_i (K S_0)_i) -------
        for (int idx = tid; idx < rows * NS; idx += nth) {
            const int i = idx / NS, j = idx % NS;
            sKS[i * lds + j] = sBeta[i] * (sV[i * lds + j] - sEg[i] * sKS[i * lds + j]);
        }
        __syncthreads();
        // ---- U = T rhs -----------------------------------------------------------
        for (int idx = tid; idx < rows * NS; idx += nth) {
            const int i = idx / NS, j = idx % NS;
            float acc = 0.f;
            for (int m = 0; m <= i; ++m) acc = fmaf(sT[i * kLdA + m], sKS[m * lds + j], acc);
            sU[i * lds + j] = acc;
        }
        __syncthreads();
        // ---- O = diag(Gamma) Q S_0 + P U ;  S <- exp(gamma_S) S_0 + K~^T U --------
        for (int idx = tid; idx < rows * NS; idx += nth) {
            const int i = idx / NS, j = idx % NS;
            float acc = sEg[i] * sQS[i * lds + j];
            for (int m = 0; m <= i; ++m) acc = fmaf(sP[i * kLdA + m], sU[m * lds + j], acc);
            store_elem(out, ((c0 + i) * p.Hv + h) * int64_t(dv) + j0 + j, acc * p.q_scale);
        }
        const float eS = sEg[rows - 1];
        for (int idx = tid; idx < dk * NS; idx += nth) {
            const int d = idx / NS, j = idx % NS;
            float acc = eS * sS[d * lds + j];
            for (int i = 0; i < rows; ++i)
                acc = fmaf(sK[i * ldq + d] * sEnd[i], sU[i * lds + j], acc);
            sS[d * lds + j] = acc;
        }
        __syncthreads();
    }

    if (p.state_out) {
        for (int idx = tid; idx < dk * NS; idx += nth) {
            const int i = idx / NS, j = idx % NS;
            p.state_out[sbase + size_t(i) * dv + j] = sS[i * lds + j];
        }
    }
}

}  // namespace

cudaError_t launch_chunk_simt(const ChunkParams& p, int dtype, cudaStream_t s) {
    const SmemLayout L = smem_layout(p.dk, p.dv);
    const dim3 grid(p.dv / L.ns, p.Hv, p.B);
    const size_t smem = L.total;
    if (p.B == 0) return cudaSuccess;
    cudaError_t e;
    if (dtype == GDN_FP32) {
        e = ensure_smem(reinterpret_cast<const void*>(chunk_simt_kernel<float>), int(smem));
        if (e != cudaSuccess) return e;
        timer_begin(s, "chunk_simt_kernel");
        chunk_simt_kernel<float><<<grid, kThreads, smem, s>>>(p);
        timer_end(s);
    } else {
        e = ensure_smem(reinterpret_cast<const void*>(chunk_simt_kernel<__nv_bfloat16>), int(smem));
        if (e != cudaSuccess) return e;
        timer_begin(s, "chunk_simt_kernel");
        chunk_simt_kernel<__nv_bfloat16><<<grid, kThreads, smem, s>>>(p);
        timer_end(s);
    }
    return cudaGetLastError();
}

}  // namespace gdn
