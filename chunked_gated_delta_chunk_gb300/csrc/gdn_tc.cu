// Tensor-core chunk kernel (bf16, dk = dv = 128) for sm_103a: tcgen05 MMAs
// with TMEM accumulators, operands in 128-byte-swizzled shared memory fed by
// TMA, the fp32 state carried in TMEM through the chunks of a sequence.
//
// Method: the chunked delta rule of "perf(qwen3_5): prefill text prompts in
// multi-token chunks" (Implementation section).  Per chunk of n <= 64 rows
// with incoming state S_0 (gamma = inclusive cumsum of g, Gamma = exp(gamma)):
//   A_ij = beta_i exp(gamma_i - gamma_j) k_i.k_j (j < i),  T = (I + A)^-1
//   U = T (diag(beta) V - diag(beta Gamma) K S_0) = U0 - W S_0,
//       U0 = T diag(beta) V,  W = T diag(beta Gamma) K
//   O = diag(Gamma) Q S_0 + (exp(gamma_t - gamma_i) q_t.k_i)_{i<=t} U
//   S_S = exp(gamma_S) S_0 + (K * exp(min(gamma_S - gamma, 0)))^T U
// T is the 64-row padded blocked inverse (8x8 Neumann blocks, then 2x2 block
// inversion level by level) in fp32 on the CUDA cores.
//
// GB300 mapping.  The state is kept transposed, Z = S^T [dv, dk], as an fp32
// TMEM accumulator (lane = value column j, column = key row d), so that every
// contraction is an M = 128 tcgen05.mma:
//   Gram     D_G  = [K; Q] K^T              (M=128, N=64, K=128)  raw q, k
//   U0^T     D_X  = V^T (T diag beta)^T     (M=128, N=64, K=64)
//   W^T      D_W  = K^T (T diag(beta Gamma r_k))^T
//   chain    D_X += Z_bf16 (-W^T)           -> v_new^T = U^T
//   output   D_O  = Z_bf16 Qs^T             Qs = diag(Gamma r_q) Q
//   state    Z   <- exp(gamma_S) Z + v_new^T Ks,  Ks = diag(exp(min(gamma_S-gamma,0)) r_k) K
//   output   D_O += v_new^T P^T             P_ti = exp(gamma_t-gamma_i) r_q,t r_k,i q_t.k_i (i<=t)
// L2 normalisation of q and k is folded into these row scalings (r = 1/|x|),
// so the Gram matrices use the raw bf16 inputs.  Every exponent is clamped at
// zero and evaluated only where its triangular mask keeps the entry.
//
// One CTA per (value head, sequence); 8 warps; warp w reads TMEM lanes
// 32 (w % 4) .. +31 and column half w / 4.  Chunk c + 1 is fetched by TMA
// while chunk c is processed (two raw stages).  Every mbarrier wait is
// bounded; on a timeout the CTA records it in a device flag, stops, and
// still frees its TMEM.
#include <cuda.h>

#include "gdn_common.cuh"
#include "gdn_tc.cuh"
#include "tc_ptx.cuh"

namespace gdn {

__device__ int g_tc_timeouts = 0;   // bumped by a CTA whose bounded wait ran out

namespace {

using namespace ptx;

constexpr int kC = 64;          // chunk rows (padded)
constexpr int kD = 128;         // dk = dv
constexpr int kThreads = 256;
constexpr uint32_t kWaitLimit = 1u << 24;
constexpr int kLdA = kC + 1;

// Shared-memory map (bytes from the 1024-aligned base).
constexpr uint32_t kStageKQ = 32768;   // [K b0 | Q b0 | K b1 | Q b1], 8 KB each
constexpr uint32_t kStageV = 16384;    // [V b0 | V b1]
constexpr uint32_t kStageBytes = kStageKQ + kStageV;
constexpr uint32_t kOffStage0 = 0;
constexpr uint32_t kOffP = 2 * kStageBytes;          // P (bf16 [t][i], K-major)      8 KB
constexpr uint32_t kOffTb = kOffP + 8192;            // T diag(beta)                   8 KB
constexpr uint32_t kOffTbg = kOffTb + 8192;          // T diag(beta Gamma r_k)         8 KB
constexpr uint32_t kOffWt = kOffTbg + 8192;          // -W^T (bf16 [d][t], MN-major)  16 KB
constexpr uint32_t kOffZ = kOffWt + 16384;           // Z bf16 [j][d] K-major         32 KB
constexpr uint32_t kOffVn = kOffZ + 32768;           // v_new^T bf16 [j][i] K-major   16 KB
constexpr uint32_t kOffA = kOffVn + 16384;           // A fp32 [64][65]
constexpr uint32_t kOffT = kOffA + kC * kLdA * 4;    // T fp32 [64][65]
constexpr uint32_t kOffTmp = kOffT + kC * kLdA * 4;  // inverse scratch, 1536 floats
constexpr uint32_t kOffVec = kOffTmp + 1536 * 4;     // 8 vectors of 64 floats
constexpr uint32_t kOffBar = kOffVec + 8 * kC * 4;   // 3 mbarriers + TMEM slot + flags
constexpr uint32_t kSmemBytes = kOffBar + 64 + 1024; // + alignment slack

// TMEM columns.
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColZ = 0;
constexpr uint32_t kColX = 128;
constexpr uint32_t kColG = 192;
constexpr uint32_t kColW = 256;
constexpr uint32_t kColO = 320;

// Offset of (row, col) in a swizzled K-major tile of 64-column blocks.
__device__ __forceinline__ uint32_t toff(int row, int col, uint32_t block_stride) {
    const int blk = col >> 6, c = col & 63;
    return uint32_t(blk) * block_stride + uint32_t(row) * 128u +
           (uint32_t(((c >> 3) ^ (row & 7))) << 4) + uint32_t(c & 7) * 2u;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ void store_chunk8(uint8_t* p, const float* v) {
    uint4 u;
    u.x = pack_bf16x2(v[0], v[1]);
    u.y = pack_bf16x2(v[2], v[3]);
    u.z = pack_bf16x2(v[4], v[5]);
    u.w = pack_bf16x2(v[6], v[7]);
    *reinterpret_cast<uint4*>(p) = u;
}

__device__ __forceinline__ void load_chunk8(const uint8_t* p, float* v) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(b[i]);
        v[2 * i] = f.x;
        v[2 * i + 1] = f.y;
    }
}

// T = (I + A)^-1 for the strictly lower 64x64 A (padded rows zero): 8x8
// diagonal blocks by (I - N)(I + N^2)(I + N^4), then 2x2 block inversion,
// level by level.  All threads of the CTA take part.
__device__ void block_inverse_64(const float* sA, float* sT, float* sTmp) {
    const int tid = threadIdx.x, nth = blockDim.x;
    const int warp = tid >> 5, lane = tid & 31;
    for (int idx = tid; idx < kC * kLdA; idx += nth) sT[idx] = 0.f;
    __syncthreads();
    if (warp < kC / 8) {
        const int o = warp * 8;
        float* N2 = sTmp + warp * 192;
        float* N4 = N2 + 64;
        float* X = N4 + 64;
        for (int e = lane; e < 64; e += 32) {
            const int r = e >> 3, c = e & 7;
            float acc = 0.f;
            for (int m = 0; m < 8; ++m) acc = fmaf(sA[(o + r) * kLdA + o + m], sA[(o + m) * kLdA + o + c], acc);
            N2[e] = acc;
        }
        __syncwarp();
        for (int e = lane; e < 64; e += 32) {
            const int r = e >> 3, c = e & 7;
            float acc = 0.f, nn2 = 0.f;
            for (int m = 0; m < 8; ++m) {
                acc = fmaf(N2[r * 8 + m], N2[m * 8 + c], acc);
                nn2 = fmaf(sA[(o + r) * kLdA + o + m], N2[m * 8 + c], nn2);
            }
            N4[e] = acc;
            X[e] = (r == c ? 1.f : 0.f) - sA[(o + r) * kLdA + o + c] + N2[e] - nn2;
        }
        __syncwarp();
        for (int e = lane; e < 64; e += 32) {
            const int r = e >> 3, c = e & 7;
            float acc = X[e];
            for (int m = 0; m < 8; ++m) acc = fmaf(X[r * 8 + m], N4[m * 8 + c], acc);
            sT[(o + r) * kLdA + o + c] = acc;
        }
    }
    __syncthreads();
    for (int size = 8; size < kC; size *= 2) {
        const int pairs = kC / (2 * size), per = size * size;
        for (int idx = tid; idx < pairs * per; idx += nth) {
            const int pr = idx / per, r = (idx / size) % size, c = idx % size;
            const int o = pr * 2 * size;
            float acc = 0.f;
            for (int m = c; m < size; ++m)
                acc = fmaf(sA[(o + size + r) * kLdA + o + m], sT[(o + m) * kLdA + o + c], acc);
            sTmp[idx] = acc;
        }
        __syncthreads();
        for (int idx = tid; idx < pairs * per; idx += nth) {
            const int pr = idx / per, r = (idx / size) % size, c = idx % size;
            const int o = pr * 2 * size;
            float acc = 0.f;
            for (int m = 0; m <= r; ++m)
                acc = fmaf(sT[(o + size + r) * kLdA + o + size + m], sTmp[pr * per + m * size + c], acc);
            sT[(o + size + r) * kLdA + o + c] = -acc;
        }
        __syncthreads();
    }
}

struct Maps {
    CUtensorMap q, k, v;
};

__global__ void __launch_bounds__(kThreads, 1)
chunk_tc_kernel(const ChunkParams p, const __grid_constant__ Maps maps) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float* sA = reinterpret_cast<float*>(sm + kOffA);
    float* sT = reinterpret_cast<float*>(sm + kOffT);
    float* sTmp = reinterpret_cast<float*>(sm + kOffTmp);
    float* vGam = reinterpret_cast<float*>(sm + kOffVec);   // gamma (cumsum)
    float* vEg = vGam + kC;                                 // Gamma = exp(gamma)
    float* vBeta = vEg + kC;
    float* vRk = vBeta + kC;                                // 1/|k_i|
    float* vRq = vRk + kC;                                  // 1/|q_t|
    float* vEnd = vRq + kC;                                 // exp(min(gamma_S - gamma_i, 0)) r_k,i
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kOffBar);   // [0,1] TMA stages, [2] MMA
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kOffBar + 24);
    int* s_err = reinterpret_cast<int*>(sm + kOffBar + 28);

    const int h = blockIdx.x, n = blockIdx.y;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3, half = warp >> 2;
    const int row = quarter * 32 + lane;                // TMEM lane owned by this thread
    const uint32_t lane_addr = uint32_t(quarter * 32) << 16;
    const int kh = h / (p.Hv / p.Hk);
    const int Hv = p.Hv;

    const __nv_bfloat16* gq = static_cast<const __nv_bfloat16*>(p.q);
    const __nv_bfloat16* gk = static_cast<const __nv_bfloat16*>(p.k);
    const __nv_bfloat16* gv = static_cast<const __nv_bfloat16*>(p.v);
    __nv_bfloat16* gout = static_cast<__nv_bfloat16*>(p.out);

    int64_t t_end_all = p.cu[p.B];
    if (t_end_all > p.t_cap) t_end_all = p.t_cap;
    int64_t t0 = p.cu[n], t1 = p.cu[n + 1];
    t0 = t0 < 0 ? 0 : (t0 > t_end_all ? t_end_all : t0);
    t1 = t1 < t0 ? t0 : (t1 > t_end_all ? t_end_all : t1);
    const int nchunks = int((t1 - t0 + p.chunk - 1) / p.chunk);

    if (tid == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        mbar_init(&bars[2], 1);
        fence_mbar_init();
        *s_err = 0;
        tma_prefetch_desc(&maps.q);
        tma_prefetch_desc(&maps.k);
        tma_prefetch_desc(&maps.v);
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tZ = tmem + kColZ, tX = tmem + kColX, tG = tmem + kColG, tW = tmem + kColW,
                   tO = tmem + kColO;

    // Chunk fetch: TMA when the 64-row box lies inside the buffers, else
    // plain loads (zero beyond the last token).  Returns true when TMA was used.
    auto tma_ok = [&](int64_t cs) { return cs + kC <= t_end_all; };
    int tma_last_issued = -1;     // thread 0 only: last chunk whose TMA was issued
    auto issue_tma = [&](int c) {
        const int st = c & 1;
        tma_last_issued = c;
        uint8_t* kq = sm + kOffStage0 + st * kStageBytes;
        uint8_t* vv = kq + kStageKQ;
        const int y = int(t0 + int64_t(c) * p.chunk);
        mbar_arrive_expect_tx(&bars[st], kStageBytes);
        tma_load_2d(kq + 0, &maps.k, &bars[st], kh * kD, y);
        tma_load_2d(kq + 16384, &maps.k, &bars[st], kh * kD + 64, y);
        tma_load_2d(kq + 8192, &maps.q, &bars[st], kh * kD, y);
        tma_load_2d(kq + 24576, &maps.q, &bars[st], kh * kD + 64, y);
        tma_load_2d(vv + 0, &maps.v, &bars[st], h * kD, y);
        tma_load_2d(vv + 8192, &maps.v, &bars[st], h * kD + 64, y);
    };
    auto manual_load = [&](int c) {
        const int st = c & 1;
        uint8_t* kq = sm + kOffStage0 + st * kStageBytes;
        uint8_t* vv = kq + kStageKQ;
        const int64_t cs = t0 + int64_t(c) * p.chunk;
        for (int idx = tid; idx < kC * 16; idx += kThreads) {      // (row, 8-col chunk)
            const int r = idx >> 4, cc = (idx & 15) * 8;
            const int64_t t = cs + r;
            uint4 zk = make_uint4(0, 0, 0, 0), zq = zk, zv = zk;
            if (t < t_end_all) {
                zk = *reinterpret_cast<const uint4*>(gk + t * p.k_stride + kh * kD + cc);
                zq = *reinterpret_cast<const uint4*>(gq + t * p.q_stride + kh * kD + cc);
                zv = *reinterpret_cast<const uint4*>(gv + t * p.v_stride + int64_t(h) * kD + cc);
            }
            *reinterpret_cast<uint4*>(kq + toff(r, cc, 16384)) = zk;
            *reinterpret_cast<uint4*>(kq + 8192 + toff(r, cc, 16384)) = zq;
            *reinterpret_cast<uint4*>(vv + toff(r, cc, 8192)) = zv;
        }
    };

    bool ok = true;
    uint32_t mma_phase = 0;
    auto wait_mma = [&]() {
        if (!mbar_wait(&bars[2], mma_phase, kWaitLimit)) ok = false;
        mma_phase ^= 1u;
        tc_fence_after();
    };
    // Make every thread agree on `ok` (a barrier is needed at this point anyway).
    auto sync_ok = [&]() {
        if (!ok) atomicExch(s_err, 1);
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        ok = (*s_err == 0);
    };

    // ---- initial state -> Z (fp32 in TMEM) and Z bf16 (shared) --------------
    {
        const size_t sb = (size_t(n) * Hv + h) * kD * kD;
        for (int cb = 0; cb < 64; cb += 16) {
            float v[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int d = half * 64 + cb + i;
                v[i] = p.state_in ? p.state_in[sb + size_t(d) * kD + row] : 0.f;
            }
            tmem_st16(tZ + lane_addr + half * 64 + cb, v);
            store_chunk8(sm + kOffZ + toff(row, half * 64 + cb, 16384), v);
            store_chunk8(sm + kOffZ + toff(row, half * 64 + cb + 8, 16384), v + 8);
        }
        tmem_st_wait();
        fence_proxy_async_smem();
    }
    if (nchunks > 0 && tid == 0 && tma_ok(t0)) issue_tma(0);
    sync_ok();

    for (int c = 0; c < nchunks && ok; ++c) {
        const int st = c & 1;
        uint8_t* kq = sm + kOffStage0 + st * kStageBytes;
        uint8_t* vv = kq + kStageKQ;
        const int64_t cs = t0 + int64_t(c) * p.chunk;
        const int rows = int(t1 - cs < p.chunk ? t1 - cs : p.chunk);

        // ---- fetch: this chunk (manual if needed), prefetch the next ------------
        const bool this_tma = tma_ok(cs);
        if (!this_tma) {
            manual_load(c);
            fence_proxy_async_smem();
        }
        if (tid == 0 && c + 1 < nchunks && tma_ok(cs + p.chunk)) {
            fence_proxy_async_smem();
            issue_tma(c + 1);
        }
        if (tid < kC) {
            const bool in = tid < rows;
            vGam[tid] = in ? p.g[(cs + tid) * Hv + h] : 0.f;
            vBeta[tid] = in ? p.beta[(cs + tid) * Hv + h] : 0.f;
        }
        if (this_tma && !mbar_wait(&bars[st], uint32_t((c >> 1) & 1), kWaitLimit)) ok = false;
        sync_ok();
        if (!ok) break;

        // ---- phase 1: cumsum, row norms; issue the Gram MMA -------------------
        if (warp == 0) {
            // inclusive scan of g over 64 rows: 2 values per lane
            float a = vGam[2 * lane], b = vGam[2 * lane + 1];
            b += a;
            float s = b;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float u = __shfl_up_sync(0xffffffffu, s, o);
                if (lane >= o) s += u;
            }
            const float excl = s - b;
            a += excl;
            b = s;
            vGam[2 * lane] = a;
            vGam[2 * lane + 1] = b;
        }
        {
            // 128 rows (K 0..63, Q 0..63): warp w takes rows 16w .. 16w+15
            for (int rr = 0; rr < 16; ++rr) {
                const int r = warp * 16 + rr;
                const int isq = r >= kC, tr = r & 63;
                const uint8_t* base = kq + (isq ? 8192 : 0);
                const int col = lane * 4;
                const uint2 u = *reinterpret_cast<const uint2*>(base + toff(tr, col, 16384));
                const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&u);
                const float2 f0 = __bfloat1622float2(b2[0]), f1 = __bfloat1622float2(b2[1]);
                float ss = f0.x * f0.x + f0.y * f0.y + f1.x * f1.x + f1.y * f1.y;
                ss = warp_sum(ss);
                if (lane == 0) {
                    const float r_ = p.l2norm ? rsqrtf(ss + p.eps) : 1.f;
                    (isq ? vRq : vRk)[tr] = r_;
                }
            }
        }
        if (tid == 0) {
            tc_fence_after();
            const uint32_t idesc = idesc_bf16(128, 64, 0, 0);
            const uint32_t base = smem_u32(kq);
            for (int s = 0; s < 8; ++s) {
                const uint32_t off = uint32_t(s >> 2) * 16384u + uint32_t(s & 3) * 32u;
                umma_f16(tG, smem_desc(base + off, 16, 1024, kSwizzle128B),
                         smem_desc(base + off, 16, 1024, kSwizzle128B), idesc, s > 0);
            }
            umma_commit(&bars[2]);
        }
        __syncthreads();
        if (tid < kC) {
            const float gm = vGam[tid];
            const float gS = vGam[rows - 1];
            vEg[tid] = expf(gm);
            vEnd[tid] = tid < rows ? expf(fminf(gS - gm, 0.f)) * vRk[tid] : 0.f;
        }
        wait_mma();
        sync_ok();
        if (!ok) break;

        // ---- phase 2: masks and decays on the Gram matrices ---------------------
        {
            float v[32];
            tmem_ld16(tG + lane_addr + half * 32, v);
            tmem_ld16(tG + lane_addr + half * 32 + 16, v + 16);
            tmem_ld_wait();
            if (row < kC) {                  // A_ij = beta_i e^{g_i - g_j} r_i r_j k_i.k_j, j < i
                const int i = row;
                const float bi = vBeta[i] * vRk[i], gi = vGam[i];
#pragma unroll
                for (int q = 0; q < 32; ++q) {
                    const int j = half * 32 + q;
                    float a = 0.f;
                    if (i < rows && j < i) a = bi * expf(fminf(gi - vGam[j], 0.f)) * vRk[j] * v[q];
                    sA[i * kLdA + j] = a;
                }
            } else {                         // P_tj = e^{g_t - g_j} r_q,t r_k,j q_t.k_j, j <= t
                const int t = row - kC;
                const float rt = vRq[t], gt = vGam[t];
                float w[32];
#pragma unroll
                for (int q = 0; q < 32; ++q) {
                    const int j = half * 32 + q;
                    w[q] = (t < rows && j <= t) ? rt * expf(fminf(gt - vGam[j], 0.f)) * vRk[j] * v[q] : 0.f;
                }
#pragma unroll
                for (int q = 0; q < 32; q += 8)
                    store_chunk8(sm + kOffP + toff(t, half * 32 + q, 8192), w + q);
            }
        }
        __syncthreads();

        // ---- phase 3: blocked inverse; T diag(beta), T diag(beta Gamma r_k) -----
        block_inverse_64(sA, sT, sTmp);
        for (int idx = tid; idx < kC * 8; idx += kThreads) {
            const int t = idx >> 3, i0 = (idx & 7) * 8;
            float a[8], b[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const int i = i0 + q;
                const float tv = sT[t * kLdA + i];
                a[q] = tv * vBeta[i];
                b[q] = a[q] * vEg[i] * vRk[i];
            }
            store_chunk8(sm + kOffTb + toff(t, i0, 8192), a);
            store_chunk8(sm + kOffTbg + toff(t, i0, 8192), b);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            const uint32_t idesc = idesc_bf16(128, 64, 1, 0);   // A MN-major, B K-major
            const uint32_t vb = smem_u32(vv), kb = smem_u32(kq);
            const uint32_t tb = smem_u32(sm + kOffTb), tbg = smem_u32(sm + kOffTbg);
            for (int s = 0; s < 4; ++s) {
                // U0^T = V^T Tb^T : A = V (rows i, cols j), B = Tb [t][i]
                umma_f16(tX, smem_desc(vb + s * 2048, 8192, 1024, kSwizzle128B),
                         smem_desc(tb + s * 32, 16, 1024, kSwizzle128B), idesc, s > 0);
                // W^T = K^T Tbg^T : A = K (rows i, cols d), B = Tbg [t][i]
                umma_f16(tW, smem_desc(kb + s * 2048, 16384, 1024, kSwizzle128B),
                         smem_desc(tbg + s * 32, 16, 1024, kSwizzle128B), idesc, s > 0);
            }
            umma_commit(&bars[2]);
        }
        wait_mma();
        sync_ok();
        if (!ok) break;

        // ---- phase 4: -W^T to shared; scale Q and K rows in place --------------
        {
            float v[32];
            tmem_ld16(tW + lane_addr + half * 32, v);
            tmem_ld16(tW + lane_addr + half * 32 + 16, v + 16);
            tmem_ld_wait();
#pragma unroll
            for (int q = 0; q < 32; ++q) v[q] = -v[q];
#pragma unroll
            for (int q = 0; q < 32; q += 8)
                store_chunk8(sm + kOffWt + toff(row, half * 32 + q, 16384), v + q);
        }
        for (int idx = tid; idx < 2 * kC * 16; idx += kThreads) {
            const int isq = idx >= kC * 16, r = (idx >> 4) & 63, cc = (idx & 15) * 8;
            uint8_t* ptr = kq + (isq ? 8192 : 0) + toff(r, cc, 16384);
            const float f = isq ? (r < rows ? vEg[r] * vRq[r] : 0.f) : vEnd[r];
            float v[8];
            load_chunk8(ptr, v);
#pragma unroll
            for (int q = 0; q < 8; ++q) v[q] *= f;
            store_chunk8(ptr, v);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            const uint32_t zb = smem_u32(sm + kOffZ), wt = smem_u32(sm + kOffWt), kb = smem_u32(kq);
            const uint32_t id_x = idesc_bf16(128, 64, 0, 1);   // B MN-major
            const uint32_t id_o = idesc_bf16(128, 64, 0, 0);
            for (int s = 0; s < 8; ++s) {
                const uint32_t za = zb + uint32_t(s >> 2) * 16384u + uint32_t(s & 3) * 32u;
                // D_X (= U0^T) += Z (-W^T)
                umma_f16(tX, smem_desc(za, 16, 1024, kSwizzle128B),
                         smem_desc(wt + s * 2048, 16384, 1024, kSwizzle128B), id_x, 1);
                // D_O = Z Qs^T : B = Qs [t][d] K-major
                const uint32_t qb = kb + 8192 + uint32_t(s >> 2) * 16384u + uint32_t(s & 3) * 32u;
                umma_f16(tO, smem_desc(za, 16, 1024, kSwizzle128B),
                         smem_desc(qb, 16, 1024, kSwizzle128B), id_o, s > 0);
            }
            umma_commit(&bars[2]);
        }
        wait_mma();
        sync_ok();
        if (!ok) break;

        // ---- phase 5: v_new^T to shared; Z <- exp(gamma_S) Z --------------------
        {
            float v[32];
            tmem_ld16(tX + lane_addr + half * 32, v);
            tmem_ld16(tX + lane_addr + half * 32 + 16, v + 16);
            tmem_ld_wait();
#pragma unroll
            for (int q = 0; q < 32; q += 8)
                store_chunk8(sm + kOffVn + toff(row, half * 32 + q, 16384), v + q);
            const float eS = vEg[rows - 1];
            for (int cb = 0; cb < 64; cb += 16) {
                float z[16];
                tmem_ld16(tZ + lane_addr + half * 64 + cb, z);
                tmem_ld_wait();
#pragma unroll
                for (int q = 0; q < 16; ++q) z[q] *= eS;
                tmem_st16(tZ + lane_addr + half * 64 + cb, z);
            }
            tmem_st_wait();
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            const uint32_t vn = smem_u32(sm + kOffVn), kb = smem_u32(kq), pb = smem_u32(sm + kOffP);
            const uint32_t id_z = idesc_bf16(128, 128, 0, 1);  // B = Ks MN-major [i][d]
            const uint32_t id_o = idesc_bf16(128, 64, 0, 0);   // B = P [t][i] K-major
            for (int s = 0; s < 4; ++s) {
                umma_f16(tZ, smem_desc(vn + s * 32, 16, 1024, kSwizzle128B),
                         smem_desc(kb + s * 2048, 16384, 1024, kSwizzle128B), id_z, 1);
                umma_f16(tO, smem_desc(vn + s * 32, 16, 1024, kSwizzle128B),
                         smem_desc(pb + s * 32, 16, 1024, kSwizzle128B), id_o, 1);
            }
            umma_commit(&bars[2]);
        }
        wait_mma();
        sync_ok();
        if (!ok) break;

        // ---- phase 6: output rows; Z bf16 for the next chunk --------------------
        {
            float v[32];
            tmem_ld16(tO + lane_addr + half * 32, v);
            tmem_ld16(tO + lane_addr + half * 32 + 16, v + 16);
            tmem_ld_wait();
#pragma unroll
            for (int q = 0; q < 32; ++q) {
                const int t = half * 32 + q;
                if (t < rows)
                    gout[((cs + t) * Hv + h) * kD + row] = __float2bfloat16_rn(v[q] * p.q_scale);
            }
            for (int cb = 0; cb < 64; cb += 16) {
                float z[16];
                tmem_ld16(tZ + lane_addr + half * 64 + cb, z);
                tmem_ld_wait();
                store_chunk8(sm + kOffZ + toff(row, half * 64 + cb, 16384), z);
                store_chunk8(sm + kOffZ + toff(row, half * 64 + cb + 8, 16384), z + 8);
            }
        }
        fence_proxy_async_smem();
        sync_ok();
    }

    // ---- final state ------------------------------------------------------------
    if (ok && p.state_out) {
        const size_t sb = (size_t(n) * Hv + h) * kD * kD;
        for (int cb = 0; cb < 64; cb += 16) {
            float z[16];
            tmem_ld16(tZ + lane_addr + half * 64 + cb, z);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i) p.state_out[sb + size_t(half * 64 + cb + i) * kD + row] = z[i];
        }
    }
    if (!ok && tid == 0) {
        atomicAdd(&g_tc_timeouts, 1);
        // Let a TMA copy still in flight land before the CTA's shared memory
        // goes away (bounded like every other wait).
        if (tma_last_issued >= 0)
            mbar_wait(&bars[tma_last_issued & 1], uint32_t((tma_last_issued >> 1) & 1), kWaitLimit);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        cudaDriverEntryPointQueryResult q;
        void* f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
    }
    return fn;
}

// 2D bf16 map over rows of `width` columns with a row pitch of `stride`
// elements; boxes of 64 x 64 with the 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, int64_t width, int64_t rows, int64_t stride) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {cuuint64_t(width), cuuint64_t(rows)};
    cuuint64_t strides[1] = {cuuint64_t(stride) * 2};
    cuuint32_t box[2] = {64, 64};
    cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_chunk_tc(const ChunkParams& p, cudaStream_t s) {
    if (p.B == 0) return cudaSuccess;
    if (encode_fn() == nullptr) return cudaErrorNotSupported;
    // Rows in the maps: the known token count, else the largest count a map
    // can describe (the kernel never issues a box past cu_seqlens[B]).
    const int64_t rows = p.t_cap != INT64_MAX ? (p.t_cap > 0 ? p.t_cap : 1) : (int64_t(1) << 31) - 1;
    Maps maps;
    if (!make_map(&maps.q, p.q, int64_t(p.Hk) * kD, rows, p.q_stride) ||
        !make_map(&maps.k, p.k, int64_t(p.Hk) * kD, rows, p.k_stride) ||
        !make_map(&maps.v, p.v, int64_t(p.Hv) * kD, rows, p.v_stride))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(chunk_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(kSmemBytes));
    if (e != cudaSuccess) return e;
    chunk_tc_kernel<<<dim3(p.Hv, p.B), kThreads, kSmemBytes, s>>>(p, maps);
    return cudaGetLastError();
}

}  // namespace gdn
