// Tensor-core chunk kernels (bf16, dk = dv = 128) for sm_103a: tcgen05 MMAs
// with TMEM accumulators and TMEM-resident A operands, B operands in
// 128-byte-swizzled shared memory fed by TMA, the fp32 state carried in TMEM
// through the chunks of a sequence (or of a segment of one).
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
// inversion level by level) in fp32 on the CUDA cores and the warp MMA.
//
// GB300 mapping.  The state is kept transposed, Z = S^T [dv, dk], as an fp32
// TMEM accumulator (lane = value column j, column = key row d), so that every
// contraction is an M = 128 tcgen05.mma:
//   Gram   [K; Q] [K; Q]^T (split preparation) or [K; Q] K^T (one pass)
//   U0^T   V^T (T diag beta)^T                T split into bf16 hi + lo
//   W^T    K^T (T diag(beta Gamma r_k))^T     T split into bf16 hi + lo
//   chain  X = Zb (-W^T), U^T = U0^T + X      Zb = bf16(Z) in TMEM
//          O = Zb Qs^T                        Qs = diag(Gamma r_q) Q
//          Z += Us^T K  (Z pre-scaled by exp(gamma_S))
//                                             Us = U diag(exp(min(gamma_S-gamma,0)) r_k),
//                                             bf16 hi + lo, in TMEM
//          O += U^T P^T                       P split into bf16 hi + lo
// L2 normalisation of q and k is folded into row scalings (r = 1/|x|).  The
// masks of A and P take the decay and both norms as one power of two per
// entry, evaluated only where the mask keeps it (with g <= 0, gamma never
// increases, so these exponents need no clamp); the state update's weights
// keep the clamp at zero of exp(min(gamma_S - gamma, 0)).
// The hi/lo splits keep the inverse's products and the state update to
// ~16 bits before they meet a bf16 operand.
//
// The kernels of this file:
//   chunk_prep_kernel   the state-independent part of every chunk, all chunks
//                       in parallel, into one record per (value head, chunk);
//   chunk_state_kernel  the chain over the records (one CTA per value head,
//                       sequence and segment pass);
//   seg_out_kernel      the segment scan's combine: each segment's incoming
//                       state and its outputs O = O' + G S_s;
//   chunk_tc_kernel     the one-kernel pass without records or a workspace
//                       (384 threads: warps 0-3 and 8-11 prepare chunk c + 1
//                       while warps 4-7 run the chain of chunk c).
// Every wait is bounded; a CTA that runs out records it in a device counter,
// lets its TMA copies land and still frees its TMEM.
#include <cuda.h>

#include "gdn_common.cuh"
#include "gdn_tc.cuh"
#include "tc_ptx.cuh"

namespace gdn {

__device__ int g_tc_timeouts = 0;   // bumped by a CTA whose bounded wait ran out

namespace {

using namespace ptx;

constexpr int kC = 64;                 // chunk rows (padded)
constexpr int kD = 128;                // dk = dv
constexpr int kThreads = 384;
constexpr uint32_t kPrepThreads = 256; // warps 0-3 and 8-11
constexpr uint32_t kChainThreads = 128;
constexpr uint32_t kBarPrep = 1, kBarChain = 2;
// mbarrier waits: attempts of at most kSuspendNs each (a short hint: a
// waiter suspended for longer can oversleep the phase change), bounded in
// total to about two seconds; the polled waits (mbar_spin) of the chunk
// chain make at most kWaitLimit polls, under a second.
constexpr uint32_t kSuspendNs = 32;
constexpr uint32_t kWaitLimit = 1u << 26;
constexpr int kLdA = kC + 4;         // fp32 row stride of A and T: 16-byte aligned rows
constexpr float kLog2e = 1.4426950408889634f;
enum : int { kModeFull = 0, kModeOffset = 1, kModeTransition = 2 };

// Shared-memory map (bytes from the 1024-aligned base).
constexpr uint32_t kStageKQ = 32768;   // [K b0 | Q b0 | K b1 | Q b1], 8 KB each
constexpr uint32_t kStageV = 16384;    // [V b0 | V b1]
constexpr uint32_t kStageBytes = kStageKQ + kStageV;
constexpr uint32_t kOffWt = 2 * kStageBytes;             // -W^T bf16 [d][t] MN-major, 16 KB
constexpr uint32_t kOffP = kOffWt + 16384;               // P [buf][hi|lo] bf16 [t][i], 4 x 8 KB
constexpr uint32_t kOffTb = kOffP + 4 * 8192;            // Tb hi, Tb lo, Tbg hi, Tbg lo, 4 x 8 KB
                                                         // (split preparation: -W^T of odd chunks)
constexpr uint32_t kOffA = kOffTb + 4 * 8192;            // A fp32 [64][68]
constexpr uint32_t kOffT = kOffA + kC * kLdA * 4;        // T fp32 [64][68]
constexpr uint32_t kOffTmp = kOffT + kC * kLdA * 4;      // inverse scratch, 1536 floats
constexpr uint32_t kOffVec = kOffTmp + 1536 * 4;         // vectors
constexpr uint32_t kVecFloats = 11 * kC + 2 * 2 * kC + 2 * kC + 2;   // prep, staging, chain
constexpr uint32_t kOffBar = kOffVec + ((kVecFloats * 4 + 127) / 128) * 128;
constexpr uint32_t kNumBars = 15;
constexpr uint32_t kSmemBytes = kOffBar + kNumBars * 8 + 32 + 1024;
static_assert(kSmemBytes <= 232448, "dynamic shared memory above the 227 KB per-block limit");

// Barrier slots.
enum : int {
    B_RAW0 = 0, B_RAW1 = 1,        // TMA tiles of a stage landed
    B_GRAM = 2, B_W = 3,           // prep MMAs done
    B_READY0 = 4, B_READY1 = 5,    // prep of a chunk published
    B_X = 6, B_Z = 7, B_O = 8,     // chain MMAs done
    B_XREAD = 9,                   // chain has read U^T out of D_X
    B_WTFREE = 10,                 // chain MMA no longer reads -W^T
    B_PFREE0 = 11, B_PFREE1 = 12,  // chain MMA no longer reads P of a buffer
    B_SFREE0 = 13, B_SFREE1 = 14   // chain no longer reads a raw stage
};

// TMEM columns.
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColZ = 0;      // fp32 Z [128 lanes x 128]
constexpr uint32_t kColZb = 128;   // bf16 pairs of Z, A operand (64 columns)
constexpr uint32_t kColX = 192;    // U0^T, then U^T (64)
constexpr uint32_t kColO = 256;    // O^T (64)
constexpr uint32_t kColGW = 320;   // Gram, then W^T (64)
constexpr uint32_t kColU = 384;    // U hi, U lo, Us hi, Us lo (4 x 32)

// The sequence whose chains the CTAs of grid row y run: the sequences in
// order of decreasing length (ties by index).  The block scheduler hands out
// CTAs in index order, so when the (sequence, head) units fill more than one
// wave the longest chains start in the first.  Every CTA derives the same
// permutation from cu_seqlens (one warp: each lane ranks one or two
// sequences); up to 64 sequences, else the identity.  Called by whole warps.
constexpr int kLongestFirstMax = 64;
__device__ __forceinline__ int seq_of_row(const int32_t* cu, int B, int y) {
    if (B <= 1 || B > kLongestFirstMax) return y;
    const int lane = threadIdx.x & 31;
    auto len = [&](int i) {
        const int a = cu[i], b = cu[i + 1];
        return b > a ? b - a : 0;
    };
    for (int base = 0; base < B; base += 32) {
        const int i = base + lane;
        int rank = -1;
        if (i < B) {
            const int li = len(i);
            rank = 0;
            for (int j = 0; j < B; ++j) {
                const int lj = len(j);
                rank += (lj > li || (lj == li && j < i)) ? 1 : 0;
            }
        }
        const unsigned m = __ballot_sync(0xffffffffu, rank == y);
        if (m) return base + __ffs(int(m)) - 1;
    }
    return y;
}

// Index arithmetic of the chain kernels in 32 bits: token indices fit
// (cu_seqlens is int32), and every thread of a CTA computes them, where the
// 64-bit divisions cost a few thousand cycles of issue.
__device__ __forceinline__ int ceil_div32(int64_t a, int b) { return int((uint32_t(a) + uint32_t(b) - 1u) / uint32_t(b)); }
// Segment slot of (sequence n starting at token t0, segment s).
__device__ __forceinline__ int64_t seg_slot32(int64_t t0, int n, int s, int64_t seg_tokens) {
    return int64_t(uint32_t(t0) / uint32_t(seg_tokens)) + n + s;
}

// Offset of (row, col) in a swizzled tile of 64-column blocks (128-byte rows).
__device__ __forceinline__ uint32_t toff(int row, int col, uint32_t block_stride) {
    const int blk = col >> 6, c = col & 63;
    return uint32_t(blk) * block_stride + uint32_t(row) * 128u +
           (uint32_t(((c >> 3) ^ (row & 7))) << 4) + uint32_t(c & 7) * 2u;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// 2^x with the hardware approximation (relative error about 2^-22; results
// below the smallest normal flush to zero).
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ void store_chunk8(uint8_t* p, const float* v) {
    uint4 u;
    u.x = pack_bf16x2(v[0], v[1]);
    u.y = pack_bf16x2(v[2], v[3]);
    u.z = pack_bf16x2(v[4], v[5]);
    u.w = pack_bf16x2(v[6], v[7]);
    *reinterpret_cast<uint4*>(p) = u;
}

// A pair (a0, a1) as bf16 hi = (bf16(a0), bf16(a1)) and lo = bf16(a - hi),
// each packed in one word: one paired conversion for hi, whose halves are
// read back as floats by shifting.
__device__ __forceinline__ void split_pair(float a0, float a1, uint32_t& hi, uint32_t& lo) {
    hi = pack_bf16x2(a0, a1);
    const float h0 = __uint_as_float(hi << 16), h1 = __uint_as_float(hi & 0xffff0000u);
    lo = pack_bf16x2(a0 - h0, a1 - h1);
}

// hi = bf16(v), lo = bf16(v - hi), 8 values each.
__device__ __forceinline__ void store_split8(uint8_t* phi, uint8_t* plo, const float* v) {
    uint4 h, l;
    split_pair(v[0], v[1], h.x, l.x);
    split_pair(v[2], v[3], h.y, l.y);
    split_pair(v[4], v[5], h.z, l.z);
    split_pair(v[6], v[7], h.w, l.w);
    *reinterpret_cast<uint4*>(phi) = h;
    *reinterpret_cast<uint4*>(plo) = l;
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

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
    uint32_t r[16], s[16];
    __syncwarp();
    GDN_TMEM_LD_X16(taddr, r);
    GDN_TMEM_LD_X16(taddr + 16, s);
    tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        v[i] = __uint_as_float(r[i]);
        v[16 + i] = __uint_as_float(s[i]);
    }
}

__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float* v) {
    uint32_t r0[16], r1[16], r2[16], r3[16];
    __syncwarp();
    GDN_TMEM_LD_X16(taddr, r0);
    GDN_TMEM_LD_X16(taddr + 16, r1);
    GDN_TMEM_LD_X16(taddr + 32, r2);
    GDN_TMEM_LD_X16(taddr + 48, r3);
    tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        v[i] = __uint_as_float(r0[i]);
        v[16 + i] = __uint_as_float(r1[i]);
        v[32 + i] = __uint_as_float(r2[i]);
        v[48 + i] = __uint_as_float(r3[i]);
    }
}

// x = hi + lo with hi, lo in tf32 (10 stored mantissa bits each, round to
// nearest away); hi + lo carries about 22 bits of x.
__device__ __forceinline__ void split_tf32(float x, uint32_t& hi, uint32_t& lo) {
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(hi) : "f"(x));
    const float r = x - __uint_as_float(hi);
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(lo) : "f"(r));
}

// d += a b for one 16x8x8 tf32 warp MMA (fp32 accumulate).  Fragment
// ownership, with g = lane / 4 and t = lane % 4: a0 (g, t), a1 (g+8, t),
// a2 (g, t+4), a3 (g+8, t+4); b0 (k=t, n=g), b1 (k=t+4, n=g);
// d0 (g, 2t), d1 (g, 2t+1), d2 (g+8, 2t), d3 (g+8, 2t+1).
__device__ __forceinline__ void mma_tf32_16x8x8(float* d, const uint32_t* a, const uint32_t* b) {
    asm volatile("mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 "
                 "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// d += a b to about fp32 accuracy from three tf32 MMAs (hi hi + hi lo + lo hi,
// the lo lo term is below fp32 rounding); the cross terms gather in e.
__device__ __forceinline__ void mma_3xtf32(float* d, float* e, const float* a, const float* b) {
    uint32_t ah[4], al[4], bh[2], bl[2];
#pragma unroll
    for (int i = 0; i < 4; ++i) split_tf32(a[i], ah[i], al[i]);
#pragma unroll
    for (int i = 0; i < 2; ++i) split_tf32(b[i], bh[i], bl[i]);
    mma_tf32_16x8x8(e, al, bh);
    mma_tf32_16x8x8(e, ah, bl);
    mma_tf32_16x8x8(d, ah, bh);
}

// One level of the 2x2 block inversion for diagonal blocks of size S: for
// every pair of inverted blocks T11, T22 with the off-diagonal block A21 of
// I + A, the lower-left block of the inverse is T21 = -T22 (A21 T11).  Both
// products run as 16x8 tiles on the warp MMA in split tf32, one tile per
// prep warp (S = 8 uses the upper 8 rows of a tile).  Inner-product steps
// that meet only the zero upper triangle of T11 or T22 are skipped.
template <int S>
__device__ __forceinline__ void level_products(const float* sA, float* sT, float* sTmp, int pw, int lane) {
    constexpr int kPairs = kC / (2 * S);
    constexpr bool kRows16 = S >= 16;
    constexpr int kRT = kRows16 ? S / 16 : 1, kCT = S / 8;
    constexpr int kTiles = kPairs * kRT * kCT;
    constexpr int kLdT = S == 8 ? 24 : S + 8;        // conflict-free B-fragment rows
    static_assert(kTiles <= int(kPrepThreads / 32), "one tile per prep warp");
    static_assert(kPairs * S * kLdT <= 1536, "tmp fits the inverse scratch");
    const int g = lane >> 2, t = lane & 3;
    const bool active = pw < kTiles;
    const int pr = pw / (kRT * kCT), rem = pw % (kRT * kCT);
    const int r0 = (rem / kCT) * 16, n0 = (rem % kCT) * 8;
    const int o = pr * 2 * S;
    float* tmp = sTmp + pr * S * kLdT;
    if (active) {
        // tmp = A21 T11 on rows r0.., columns n0..; T11[m][n] = 0 for m < n
        float d[4] = {0.f, 0.f, 0.f, 0.f}, e[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int k0 = 0; k0 < S; k0 += 8) {
            if (k0 < n0) continue;
            const float* ar = sA + (o + S + r0 + g) * kLdA + o + k0 + t;
            const float* br = sT + (o + k0 + t) * kLdA + o + n0 + g;
            const float a[4] = {ar[0], kRows16 ? ar[8 * kLdA] : 0.f, ar[4], kRows16 ? ar[8 * kLdA + 4] : 0.f};
            const float b[2] = {br[0], br[4 * kLdA]};
            mma_3xtf32(d, e, a, b);
        }
        *reinterpret_cast<float2*>(tmp + (r0 + g) * kLdT + n0 + 2 * t) = make_float2(d[0] + e[0], d[1] + e[1]);
        if (kRows16)
            *reinterpret_cast<float2*>(tmp + (r0 + g + 8) * kLdT + n0 + 2 * t) = make_float2(d[2] + e[2], d[3] + e[3]);
    }
    named_sync(kBarPrep, kPrepThreads);
    if (active) {
        // T21 = -T22 tmp on rows r0.., columns n0..; T22[r][m] = 0 for m > r
        float d[4] = {0.f, 0.f, 0.f, 0.f}, e[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int k0 = 0; k0 < S; k0 += 8) {
            if (k0 >= r0 + 16) continue;
            const float* ar = sT + (o + S + r0 + g) * kLdA + o + S + k0 + t;
            const float* br = tmp + (k0 + t) * kLdT + n0 + g;
            const float a[4] = {ar[0], kRows16 ? ar[8 * kLdA] : 0.f, ar[4], kRows16 ? ar[8 * kLdA + 4] : 0.f};
            const float b[2] = {br[0], br[4 * kLdT]};
            mma_3xtf32(d, e, a, b);
        }
        float* out = sT + (o + S + r0 + g) * kLdA + o + n0 + 2 * t;
        *reinterpret_cast<float2*>(out) = make_float2(-(d[0] + e[0]), -(d[1] + e[1]));
        if (kRows16) *reinterpret_cast<float2*>(out + 8 * kLdA) = make_float2(-(d[2] + e[2]), -(d[3] + e[3]));
    }
    named_sync(kBarPrep, kPrepThreads);
}

// T = (I + A)^-1 for the strictly lower 64x64 A (padded rows zero): 8x8
// diagonal blocks by (I - N)(I + N^2)(I + N^4), then 2x2 block inversion,
// level by level.  Run by the 256 prep threads (index pt) with named barriers.
__device__ void block_inverse_64(const float* sA, float* sT, float* sTmp, int pt) {
    const int pw = pt >> 5, lane = pt & 31;
    {
        // 8 prep warps, one 8x8 diagonal block each.  Lane owns rows r and
        // r + 4 of column c (r = lane >> 3, c = lane & 7); matrices of the
        // block are exchanged through per-warp scratch in shared memory.
        const int o = pw * 8;
        const int r = lane >> 3, c = lane & 7;
        float* W0 = sTmp + pw * 192;      // N^2, then N^4
        float* W1 = W0 + 64;              // X = (I - N)(I + N^2)
        float nrow[2][8], ncol[8];
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            nrow[0][m] = sA[(o + r) * kLdA + o + m];
            nrow[1][m] = sA[(o + r + 4) * kLdA + o + m];
            ncol[m] = sA[(o + m) * kLdA + o + c];
        }
        float n2[2];
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
            float acc = 0.f;
#pragma unroll
            for (int m = 0; m < 8; ++m) acc = fmaf(nrow[h2][m], ncol[m], acc);
            n2[h2] = acc;
            W0[(r + 4 * h2) * 8 + c] = acc;
        }
        __syncwarp();
        float n2row[2][8], n2col[8];
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            n2row[0][m] = W0[r * 8 + m];
            n2row[1][m] = W0[(r + 4) * 8 + m];
            n2col[m] = W0[m * 8 + c];
        }
        float n4[2], x[2];
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
            float a4 = 0.f, nn2 = 0.f;
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                a4 = fmaf(n2row[h2][m], n2col[m], a4);
                nn2 = fmaf(nrow[h2][m], n2col[m], nn2);
            }
            n4[h2] = a4;
            // X = (I - N)(I + N^2) = I - N + N^2 - N N^2
            x[h2] = ((r + 4 * h2) == c ? 1.f : 0.f) - sA[(o + r + 4 * h2) * kLdA + o + c] + n2[h2] - nn2;
        }
        __syncwarp();
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
            W0[(r + 4 * h2) * 8 + c] = n4[h2];
            W1[(r + 4 * h2) * 8 + c] = x[h2];
        }
        __syncwarp();
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
            float acc = x[h2];                 // X (I + N^4)
#pragma unroll
            for (int m = 0; m < 8; ++m) acc = fmaf(W1[(r + 4 * h2) * 8 + m], W0[m * 8 + c], acc);
            sT[(o + r + 4 * h2) * kLdA + o + c] = acc;
        }
    }
    named_sync(kBarPrep, kPrepThreads);
    level_products<8>(sA, sT, sTmp, pw, lane);
    level_products<16>(sA, sT, sTmp, pw, lane);
    level_products<32>(sA, sT, sTmp, pw, lane);
}

struct Maps {
    CUtensorMap q, k, v;
    CUtensorMap o;            // the output (chunk records or segments: tile stores)
    CUtensorMap g;            // the output map G of the segment scan (bf16, laid out like o)
};

// ---- split preparation ------------------------------------------------------
// Everything of a chunk that does not depend on the incoming state (norms,
// cumsum, the masked Gram matrices, the blocked inverse, U0 and W, the
// intra-chunk output weights P and the scaled queries) is solved by
// chunk_prep_kernel for all chunks at once, one CTA per (chunk slot, value
// head), two CTAs per SM.  It stores one record per chunk:
//   WQ     the B operand of the state pass's first product as it lies in
//          shared memory: for each 64-column block of d, 128 rows of bf16,
//          K-major with the 128-byte swizzle, -W [64 rows i] and
//          Qs = diag(Gamma r_q) Q [64 rows t]; -W first when the chunk is an
//          even chunk of the pass that reads it, Qs first for an odd one,
//   P      hi and lo images [64][64] bf16 (same layout),
//   U0^T   the TMEM fragments of the 256 preparing threads, 32 fp32 each,
//          stored in 16-byte groups interleaved across a warp's lanes, so that
//          a thread of the state pass reads its lane's columns coalesced,
//   vec    end weights e_i = exp(min(gamma_S - gamma_i, 0)) r_k,i and
//          exp(gamma_S).
// The state kernel (chunk_state_kernel) then streams the records instead of
// solving them.
constexpr uint32_t kRecWQ = 0;
constexpr uint32_t kRecP = 32768;
constexpr uint32_t kRecU = 49152;
constexpr uint32_t kRecVec = 81920;
static_assert(kRecVec + 512 == kPrepRecordBytes, "record layout");

// Shared-memory map of the preparation kernel (bytes from the 1024-aligned
// base).  A lives under Tb: the inverse has read A for the last time before
// Tb is written.  The P images are staged after A (and stored from there
// before Tb is written), the -W^T image in T's place and the U0^T fragments
// in Tb's once the MMAs are done; one thread stores staged images with bulk
// copies, so the record writes are whole lines.
constexpr uint32_t kPOffKQ = 0;                          // K b0 | Q b0 | K b1 | Q b1
constexpr uint32_t kPOffV = kStageKQ;                    // V b0 | V b1
constexpr uint32_t kPOffTb = kPOffV + 16384;             // Tb hi, lo, Tbg hi, lo (A first)
constexpr uint32_t kPOffPst = kPOffTb + kC * kLdA * 4;   // P hi | lo staging, after A
constexpr uint32_t kPOffT = kPOffPst + 16384;
constexpr uint32_t kPOffTmp = kPOffT + kC * kLdA * 4;
constexpr uint32_t kPOffVec = kPOffTmp + 1536 * 4;
constexpr uint32_t kPOffBar = kPOffVec + 11 * kC * 4;
constexpr int kPrepRing = 32;                            // items one lookup finds (one per lane)
constexpr uint32_t kPOffRing = kPOffBar + 3 * 8 + 8;     // the CTA's next items: kPrepRing x 32 B
constexpr uint32_t kPOffRingIdx = kPOffRing + kPrepRing * 32;   // their item numbers, then count, next candidate
constexpr int kPrepSeqs = 64;                            // sequences whose bounds sit in shared memory
constexpr uint32_t kPOffSeq = kPOffRingIdx + kPrepRing * 8 + 16;   // first token, first slot: 2 x (kPrepSeqs + 1)
constexpr uint32_t kPrepSmemBytes = kPOffSeq + 2 * (kPrepSeqs + 1) * 4 + 8 + 1024;
constexpr uint32_t kPrepTmemCols = 256;                  // Gram [K; Q][K; Q]^T (128), then W^T (64); U0^T (64)
static_assert(kC * kLdA * 4 <= 4 * 8192 && kPOffT >= kPOffTb + 4 * 8192, "A and the P staging beside Tb");
static_assert(kC * kLdA * 4 >= 16384, "-W^T staging fits in T's place");
static_assert(2 * (kPrepSmemBytes + 1024) <= 233472, "two preparation CTAs per SM");

// Persistent: each CTA takes items (value head, chunk slot) with a grid
// stride and prefetches the next item's raw tiles (TMA) and g, beta while
// it finishes the current one, so neither the setup (barriers, TMEM) nor the
// load latency is paid per chunk.
__global__ void __launch_bounds__(kPrepThreads, 2)
chunk_prep_kernel(const ChunkParams p, const __grid_constant__ Maps maps) {
    griddep_wait();   // everything the grid before wrote (inputs, the records it may still read)
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* kq = sm + kPOffKQ;
    uint8_t* vv = sm + kPOffV;
    float* sA = reinterpret_cast<float*>(sm + kPOffTb);
    float* sT = reinterpret_cast<float*>(sm + kPOffT);
    float* sTmp = reinterpret_cast<float*>(sm + kPOffTmp);
    float* vGam = reinterpret_cast<float*>(sm + kPOffVec);   // g, then gamma * log2(e)
    float* vEg = vGam + kC;                                 // Gamma
    float* vBeta = vEg + kC;
    float* vRk = vBeta + kC;                                // 1/|k_i|
    float* vRq = vRk + kC;                                  // 1/|q_t|
    float* vEnd = vRq + kC;                                 // e_i
    float* vFb = vEnd + kC;                                 // beta_i
    float* vFbg = vFb + kC;                                 // beta_i Gamma_i r_k,i
    float* vCol = vFbg + kC;                                // gamma_j - log2 r_k,j (log2 domain)
    float* vRowA = vCol + kC;                               // gamma_i + log2 r_k,i
    float* vRowP = vRowA + kC;                              // gamma_t + log2 r_q,t
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kPOffBar);   // raw tiles, Gram, U0 / W
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kPOffBar + 24);

    const int pt = threadIdx.x, pw = pt >> 5, lane = pt & 31;
    const int phalf = pw >> 2;                              // column half of TMEM reads
    const int row = (pw & 3) * 32 + lane;                   // TMEM lane of this thread
    const uint32_t lane_addr = uint32_t((pw & 3) * 32) << 16;
    const int Hv = p.Hv;
    const int64_t n_items = p.prep_slots * int64_t(Hv);

    int64_t t_end_all = p.cu[p.B];
    if (t_end_all > p.t_cap) t_end_all = p.t_cap;
    auto seq_first = [&](int m) {
        const int64_t t = p.cu[m];
        return t < 0 ? int64_t(0) : (t > t_end_all ? t_end_all : t);
    };
    // The chunk of item = h * prep_slots + slot: the last sequence n with
    // t0_n / chunk + n <= slot, chunk c = slot - (t0_n / chunk + n); false
    // when the slot holds no chunk.
    // odd: the chunk is an odd chunk of the state pass that reads it (its
    // segment's passes with the segment scan, else the whole sequence), which
    // fixes the order of the record's WQ tile.
    struct Item {
        int h, slot, rows;
        int64_t cs;
        bool tma, odd;
    };
    const bool segmented = p.seg_chunks > 0 && p.seg_max >= 2;
    // Each sequence's first token and first chunk slot (t0_n / chunk + n),
    // from shared memory for up to kPrepSeqs sequences, else from cu_seqlens.
    // Items, slots and token indices fit in 32 bits (the host runs this
    // kernel only when Hv * prep_slots < 2^31; cu_seqlens is int32).
    int32_t* s_first = reinterpret_cast<int32_t*>(sm + kPOffSeq);
    int32_t* s_slot0 = s_first + kPrepSeqs + 1;
    const bool seq_table = p.B <= kPrepSeqs;
    if (seq_table && pt <= p.B) {
        const int32_t t = int32_t(seq_first(pt));
        s_first[pt] = t;
        s_slot0[pt] = int32_t(uint32_t(t) / uint32_t(p.chunk)) + pt;
    }
    __syncthreads();
    auto first_of = [&](int m) { return seq_table ? int64_t(s_first[m]) : seq_first(m); };
    auto slot0_of = [&](int m) {
        return seq_table ? int64_t(s_slot0[m]) : int64_t(uint32_t(seq_first(m)) / uint32_t(p.chunk)) + m;
    };
    auto resolve = [&](int64_t item, Item& it) {
        const uint32_t slots = uint32_t(p.prep_slots), chunk = uint32_t(p.chunk);
        it.h = int(uint32_t(item) / slots);
        it.slot = int(uint32_t(item) - uint32_t(it.h) * slots);
        int lo = 0, hi = p.B - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (slot0_of(mid) <= it.slot) lo = mid;
            else hi = mid - 1;
        }
        const int64_t t0 = first_of(lo);
        int64_t t1 = first_of(lo + 1);                    // cu_seqlens[lo + 1] clamped to [t0, T]
        t1 = t1 < t0 ? t0 : t1;
        const int64_t c = int64_t(it.slot) - slot0_of(lo);
        if (c < 0 || c * chunk >= t1 - t0) return false;
        it.cs = t0 + c * chunk;
        it.rows = int(t1 - it.cs < int64_t(chunk) ? t1 - it.cs : int64_t(chunk));
        it.tma = it.cs + kC <= t_end_all;
        uint32_t local = uint32_t(c);
        if (segmented) {
            const uint32_t L = uint32_t(p.seg_chunks);
            const uint32_t seq_chunks = (uint32_t(t1 - t0) + chunk - 1) / chunk;
            const uint32_t short_by = ((seq_chunks + L - 1) / L) * L - seq_chunks;
            const uint32_t seg = (local + short_by) / L;
            local -= seg == 0 ? 0u : seg * L - short_by;
        }
        it.odd = (local & 1) != 0;
        return true;
    };
    // The CTA's items are blockIdx.x + k * gridDim.x that hold a chunk.  The
    // last warp looks up the next kPrepRing candidates at once, one per lane,
    // and packs those that hold a chunk into a ring in shared memory; the
    // items are then read from the ring (a lookup costs a thread about 1K
    // cycles, too much to make once per item).
    static_assert(sizeof(Item) <= 32, "an item's place in the ring");
    Item* ring = reinterpret_cast<Item*>(sm + kPOffRing);
    int64_t* ring_idx = reinterpret_cast<int64_t*>(sm + kPOffRingIdx);
    int* ring_n = reinterpret_cast<int*>(ring_idx + kPrepRing);
    int64_t* ring_cand = ring_idx + kPrepRing + 1;
    auto fill_ring = [&](int64_t cand) {          // the last warp, all lanes
        int n = 0;
        while (n == 0 && cand < n_items) {
            const int64_t idx = cand + int64_t(lane) * gridDim.x;
            Item it;
            const bool ok = idx < n_items && resolve(idx, it);
            const uint32_t m = __ballot_sync(0xffffffffu, ok);
            if (ok) {
                const int pos = __popc(m & ((1u << lane) - 1u));
                ring[pos] = it;
                ring_idx[pos] = idx;
            }
            n = __popc(m);
            cand += int64_t(kPrepRing) * gridDim.x;
        }
        if (lane == 0) {
            *ring_n = n;
            *ring_cand = cand;
        }
    };
    auto prefetch_box = [&](const Item& it, int b) {   // box b of K (0, 1), Q (2, 3), V (4, 5) toward L2
        const CUtensorMap* map = b < 2 ? &maps.k : (b < 4 ? &maps.q : &maps.v);
        const int head = b < 4 ? it.h / (Hv / p.Hk) : it.h;
        tma_prefetch_2d(map, head * kD + (b & 1) * 64, int(it.cs));
    };
    auto issue_raw = [&](const Item& it) {      // thread 0: the 64-row boxes of K, Q, V
        const int kh = it.h / (Hv / p.Hk);
        const int y = int(it.cs);
        mbar_arrive_expect_tx(&bars[0], kStageBytes);
        tma_load_2d(kq + 0, &maps.k, &bars[0], kh * kD, y);
        tma_load_2d(kq + 16384, &maps.k, &bars[0], kh * kD + 64, y);
        tma_load_2d(kq + 8192, &maps.q, &bars[0], kh * kD, y);
        tma_load_2d(kq + 24576, &maps.q, &bars[0], kh * kD + 64, y);
        tma_load_2d(vv + 0, &maps.v, &bars[0], it.h * kD, y);
        tma_load_2d(vv + 8192, &maps.v, &bars[0], it.h * kD + 64, y);
    };

    if (pw == kPrepThreads / 32 - 1) fill_ring(blockIdx.x);
    __syncthreads();
    int rn = *ring_n, rp = 0;                               // items in the ring, the current one's place
    if (rn == 0) return;                                    // no chunk for this CTA
    Item cur = ring[0];
    int64_t item = ring_idx[0];
    if (pt == 0) {
        for (int i = 0; i < 3; ++i) mbar_init(&bars[i], 1);
        fence_mbar_init();
        tma_prefetch_desc(&maps.q);
        tma_prefetch_desc(&maps.k);
        tma_prefetch_desc(&maps.v);
        if (cur.tma) issue_raw(cur);
    }
    // g, beta of the current item (rows past the chunk are zero)
    float g_in = 0.f, b_in = 0.f;
    if (pt < cur.rows) {
        g_in = p.g[(cur.cs + pt) * Hv + cur.h];
        b_in = p.beta[(cur.cs + pt) * Hv + cur.h];
    }
    __syncwarp();
    if (pw == 0) {
        tmem_alloc(tmem_slot, kPrepTmemCols);
        tmem_relinquish();
    }
    for (int idx = pt; idx < kC * kLdA; idx += kPrepThreads) sT[idx] = 0.f;   // upper triangle stays 0
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tGW = tmem, tX = tmem + 128;
    uint32_t raw_phase = 0, mma_phase = 0;                 // completed phases of bars[0], of bars[1] / bars[2]
    bool raw_pending = cur.tma, fail = false;
    while (item < n_items) {
        const int h = cur.h, rows = cur.rows;
        const int kh = h / (Hv / p.Hk);
        const int64_t cs = cur.cs;
        uint8_t* rec = p.prep_ws + (size_t(h) * size_t(p.prep_slots) + size_t(cur.slot)) * kPrepRecordBytes;
        if (pt < kC) {
            vGam[pt] = g_in;
            vBeta[pt] = b_in;
        }
        // ---- raw tiles: TMA when the whole 64-row box lies inside the buffers,
        // else plain loads (rows past the buffers are zero)
        if (!cur.tma) {
            const __nv_bfloat16* gq = static_cast<const __nv_bfloat16*>(p.q);
            const __nv_bfloat16* gk = static_cast<const __nv_bfloat16*>(p.k);
            const __nv_bfloat16* gv = static_cast<const __nv_bfloat16*>(p.v);
            for (int idx = pt; idx < kC * 16; idx += kPrepThreads) {
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
            fence_proxy_async_smem();
        }
        bool lf = false;
        if (cur.tma && pt == 0) lf = !mbar_wait(&bars[0], raw_phase & 1, kWaitLimit, kSuspendNs);
        if (__syncthreads_or(lf)) { fail = true; break; }
        if (cur.tma) {
            ++raw_phase;
            raw_pending = false;
        }
        // ---- Gram MMA [K; Q] [K; Q]^T (its diagonal gives the row norms); ------
        // ---- cumsum of g (log2 domain) while it runs ----------------------------
        tc_fence_after();
        if (pt == 32) {
            const uint32_t id_gram = idesc_bf16(128, 128, 0, 0);
            const uint64_t d0 = smem_desc(smem_u32(kq), 16, 1024, kSwizzle128B);
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                const uint32_t off = uint32_t(s >> 2) * 16384u + uint32_t(s & 3) * 32u;
                umma_f16(tGW, d0 + (off >> 4), d0 + (off >> 4), id_gram, s > 0);
            }
            umma_commit(&bars[1]);
        }
        __syncwarp();
        if (pw == 0) {
            float a = vGam[2 * lane], bb = vGam[2 * lane + 1];
            bb += a;
            float s = bb;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float u = __shfl_up_sync(0xffffffffu, s, o);
                if (lane >= o) s += u;
            }
            a += s - bb;
            vGam[2 * lane] = a * kLog2e;
            vGam[2 * lane + 1] = s * kLog2e;
        }
        // the next item comes from the ring, which the last warp refills when
        // this item is its last.  While the Gram product runs, warps 2-7 (idle
        // here) send the next item's six tile boxes toward L2, one each: a
        // prefetch holds its thread a few hundred cycles
        const bool refill = rp + 1 >= rn;
        if (refill) {
            if (pw == kPrepThreads / 32 - 1) {
                fill_ring(*ring_cand);
                __syncwarp();
                if (lane < 6 && *ring_n > 0 && ring[0].tma) prefetch_box(ring[0], lane);
            }
        } else if (pw >= 2 && lane == 0 && ring[rp + 1].tma) {
            prefetch_box(ring[rp + 1], pw - 2);
        }
        if (pt == 0) {
            lf = !mbar_wait(&bars[1], mma_phase & 1, kWaitLimit, kSuspendNs);
            bulk_wait_group_read<0>();                    // the last item's staged images are read
        }
        if (__syncthreads_or(lf)) { fail = true; break; }
        // the next item, and its g, beta into registers: needed once this
        // item's products have read the tiles
        if (refill) {
            rn = *ring_n;
            rp = -1;
        }
        const int np = rp + 1;
        const Item nxt = np < rn ? ring[np] : cur;
        const int64_t next = np < rn ? ring_idx[np] : n_items;
        float g_nx = 0.f, b_nx = 0.f;
        if (next < n_items && pt < nxt.rows) {
            g_nx = p.g[(nxt.cs + pt) * Hv + nxt.h];
            b_nx = p.beta[(nxt.cs + pt) * Hv + nxt.h];
        }
        tc_fence_after();
        if (phalf == 0) {
            // row norms: |k_i|^2 and |q_t|^2 on the diagonal (TMEM lane r, column r)
            uint32_t d[32];
            __syncwarp();
            GDN_TMEM_LD_X16(tGW + lane_addr + (pw & 3) * 32, d);
            GDN_TMEM_LD_X16(tGW + lane_addr + (pw & 3) * 32 + 16, (d + 16));
            tmem_ld_wait();
            float ss = 0.f;
#pragma unroll
            for (int k = 0; k < 32; ++k) ss = k == lane ? __uint_as_float(d[k]) : ss;
            const float r = p.l2norm ? rsqrtf(ss + p.eps) : 1.f;
            if (row < kC) vRk[row] = r;
            else vRq[row - kC] = r;
        }
        __syncthreads();
        if (pt < kC) {
            const float gm = vGam[pt];
            const float eg = exp2f(gm);
            vEg[pt] = eg;
            const float e = pt < rows ? exp2f(fminf(vGam[rows - 1] - gm, 0.f)) * vRk[pt] : 0.f;
            vEnd[pt] = e;
            vFb[pt] = vBeta[pt];
            vFbg[pt] = vBeta[pt] * eg * vRk[pt];
            // the masks' decays and row norms as one power of two per entry:
            // exp(gamma_i - gamma_j) r_i r_j = 2^(row_i - col_j)
            const float lk = log2f(vRk[pt]);
            vCol[pt] = gm - lk;
            vRowA[pt] = gm + lk;
            vRowP[pt] = gm + log2f(vRq[pt]);
            reinterpret_cast<float*>(rec + kRecVec)[pt] = e;
            if (pt == rows - 1) reinterpret_cast<float*>(rec + kRecVec)[kC] = eg;
        }
        // ---- masks and decays on the Gram matrices: A to shared, P to the record
        __syncthreads();
        if (mma_phase > 0)                                // T's place held the last -W^T image: T = 0 again
            for (int idx = pt; idx < kC * kLdA / 4; idx += kPrepThreads)
                reinterpret_cast<float4*>(sT)[idx] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (phalf == 1 && (pw & 1) == 0) {
            // warps 4 and 6: rows 0-31 of A and of P against columns 32-63,
            // every entry masked (j > i, j > t)
            const int r0 = row & (kC - 1);
            if (row < kC) {
#pragma unroll
                for (int q = 0; q < 32; q += 4)
                    *reinterpret_cast<float4*>(sA + r0 * kLdA + 32 + q) = make_float4(0.f, 0.f, 0.f, 0.f);
            } else {
                const uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                for (int q = 0; q < 32; q += 8) {
                    const uint32_t o = toff(r0, 32 + q, 8192);
                    *reinterpret_cast<uint4*>(sm + kPOffPst + o) = z;
                    *reinterpret_cast<uint4*>(sm + kPOffPst + 8192 + o) = z;
                }
            }
        } else {
            float v[32];
            tmem_ld32(tGW + lane_addr + phalf * 32, v);
            // A_ij = beta_i exp(gamma_i - gamma_j) r_i r_j k_i.k_j (j < i) and
            // P_tj = exp(gamma_t - gamma_j) r_t r_j q_t.k_j (j <= t); the
            // exponents need no clamp, as g <= 0 makes gamma non-increasing
            if (row < kC) {
                const int i = row;
                const float bi = vBeta[i], ai = vRowA[i];
#pragma unroll
                for (int q = 0; q < 32; q += 4) {
                    const float4 c4 = *reinterpret_cast<const float4*>(vCol + phalf * 32 + q);
                    const float cj[4] = {c4.x, c4.y, c4.z, c4.w};
                    float a4[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int j = phalf * 32 + q + u;
                        a4[u] = (i < rows && j < i) ? bi * (v[q + u] * fast_exp2(ai - cj[u])) : 0.f;
                    }
                    *reinterpret_cast<float4*>(sA + i * kLdA + phalf * 32 + q) = make_float4(a4[0], a4[1], a4[2], a4[3]);
                }
            } else {
                const int t = row - kC;
                const float at = vRowP[t];
#pragma unroll
                for (int q = 0; q < 32; q += 4) {
                    const float4 c4 = *reinterpret_cast<const float4*>(vCol + phalf * 32 + q);
                    const float cj[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int j = phalf * 32 + q + u;
                        v[q + u] = (t < rows && j <= t) ? v[q + u] * fast_exp2(at - cj[u]) : 0.f;
                    }
                }
#pragma unroll
                for (int q = 0; q < 32; q += 8) {
                    const uint32_t o = toff(t, phalf * 32 + q, 8192);
                    store_split8(sm + kPOffPst + o, sm + kPOffPst + 8192 + o, v + q);
                }
            }
        }
        fence_proxy_async_smem();
        __syncthreads();
        if (pt == 0) {
            bulk_store(rec + kRecP, sm + kPOffPst, 16384);
            bulk_commit_group();
        }
        // ---- blocked inverse; T diag(beta), T diag(beta Gamma r_k) as hi + lo --
        block_inverse_64(sA, sT, sTmp, pt);
        if (pt == 0) bulk_wait_group_read<0>();             // the P staging, which Tb overlaps
        __syncthreads();
        // A warp takes 32 rows of one 8-column group: the groups above the
        // diagonal (T is lower triangular) are zeros, written without the
        // arithmetic
        for (int idx = pt; idx < kC * 8; idx += kPrepThreads) {
            const int t = idx & (kC - 1), i0 = (idx >> 6) * 8;
            const uint32_t o = toff(t, i0, 8192);
            if (i0 > (t | 31)) {                           // the warp's every row lies above the group
                const uint4 z = make_uint4(0u, 0u, 0u, 0u);
                *reinterpret_cast<uint4*>(sm + kPOffTb + o) = z;
                *reinterpret_cast<uint4*>(sm + kPOffTb + 8192 + o) = z;
                *reinterpret_cast<uint4*>(sm + kPOffTb + 16384 + o) = z;
                *reinterpret_cast<uint4*>(sm + kPOffTb + 24576 + o) = z;
                continue;
            }
            float a[8], bg[8], fb[8], fbg[8], tr[8];
            *reinterpret_cast<float4*>(fb) = *reinterpret_cast<const float4*>(vFb + i0);
            *reinterpret_cast<float4*>(fb + 4) = *reinterpret_cast<const float4*>(vFb + i0 + 4);
            *reinterpret_cast<float4*>(fbg) = *reinterpret_cast<const float4*>(vFbg + i0);
            *reinterpret_cast<float4*>(fbg + 4) = *reinterpret_cast<const float4*>(vFbg + i0 + 4);
            *reinterpret_cast<float4*>(tr) = *reinterpret_cast<const float4*>(sT + t * kLdA + i0);
            *reinterpret_cast<float4*>(tr + 4) = *reinterpret_cast<const float4*>(sT + t * kLdA + i0 + 4);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                a[q] = tr[q] * fb[q];
                bg[q] = tr[q] * fbg[q];
            }
            store_split8(sm + kPOffTb + o, sm + kPOffTb + 8192 + o, a);
            store_split8(sm + kPOffTb + 16384 + o, sm + kPOffTb + 24576 + o, bg);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        if (pt == 0) {
            tc_fence_after();
            const uint32_t id_uw = idesc_bf16(128, 64, 1, 0);   // A MN-major, B K-major
            const uint64_t dTb = smem_desc(smem_u32(sm + kPOffTb), 16, 1024, kSwizzle128B);
            const uint64_t dV = smem_desc(smem_u32(vv), 8192, 1024, kSwizzle128B);
            const uint64_t dK = smem_desc(smem_u32(kq), 16384, 1024, kSwizzle128B);
#pragma unroll
            for (int part = 0; part < 2; ++part)
#pragma unroll
                for (int s = 0; s < 4; ++s) {
                    // U0^T = V^T Tb^T ;  W^T = K^T Tbg^T
                    umma_f16(tX, dV + uint64_t(s * 2048 >> 4), dTb + uint64_t((part * 8192 + s * 32) >> 4), id_uw,
                             part > 0 || s > 0);
                    umma_f16(tGW, dK + uint64_t(s * 2048 >> 4), dTb + uint64_t((16384 + part * 8192 + s * 32) >> 4),
                             id_uw, part > 0 || s > 0);
                }
            umma_commit(&bars[2]);
        }
        __syncwarp();
        // ---- while U0 and W run: Qs = diag(Gamma r_q) Q to the record ----------
        for (int idx = pt; idx < kC * 16; idx += kPrepThreads) {
            const int r = idx >> 4, cc = (idx & 15) * 8;
            const float f = r < rows ? vEg[r] * vRq[r] : 0.f;
            float v[8];
            load_chunk8(kq + 8192 + toff(r, cc, 16384), v);
#pragma unroll
            for (int q = 0; q < 8; ++q) v[q] *= f;
            store_chunk8(rec + kRecWQ + (cur.odd ? 0u : 8192u) + toff(r, cc, 16384), v);
        }
        if (pt == 0) lf = !mbar_wait(&bars[2], mma_phase & 1, kWaitLimit, kSuspendNs);
        if (__syncthreads_or(lf)) { fail = true; break; }
        ++mma_phase;
        tc_fence_after();
        // ---- raw tiles are free: fetch the next item's while this one is stored
        if (next < n_items) {
            if (pt == 0 && nxt.tma) issue_raw(nxt);
            raw_pending = nxt.tma;
            g_in = g_nx;
            b_in = b_nx;
        }
        {
            // -W, K-major ([64 rows i][128 columns d], two 64-column blocks):
            // W^T (lane d, column i) read as MMA-ordered fragments and stored
            // transposed
            uint32_t r[4][8];
            const int quarter = pw & 3;
#pragma unroll
            for (int u = 0; u < 4; ++u)
                tmem_ld_16x256b_x2(tGW + (uint32_t(quarter * 32 + 16 * (u >> 1)) << 16) +
                                       uint32_t(phalf * 32 + 16 * (u & 1)),
                                   r[u]);
            tmem_ld_wait();
            const int m = lane >> 3, rr = lane & 7;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                uint32_t f[4];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    f[e] = pack_bf16x2(-__uint_as_float(r[u][2 * e]), -__uint_as_float(r[u][2 * e + 1]));
                const int i = phalf * 32 + 16 * (u & 1) + 8 * (m >> 1) + rr;
                const int d = quarter * 32 + 16 * (u >> 1) + 8 * (m & 1);
                stmatrix_x4_trans(smem_u32(sm + kPOffT + toff(i, d, 8192)), f);
            }
            // U0^T straight to the record: this thread's 32 columns as eight
            // 16-byte groups interleaved across the warp's lanes
            float v[32];
            tmem_ld32(tX + lane_addr + phalf * 32, v);
            float4* u = reinterpret_cast<float4*>(rec + kRecU) + pw * 8 * 32 + lane;
#pragma unroll
            for (int i = 0; i < 8; ++i) u[i * 32] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();                                   // TMEM read, vectors free for the next item
        if (pt == 0) {
            const uint32_t w_at = cur.odd ? 8192u : 0u;     // -W's rows in each 128-row block
            bulk_store(rec + kRecWQ + w_at, sm + kPOffT, 8192);
            bulk_store(rec + kRecWQ + 16384 + w_at, sm + kPOffT + 8192, 8192);
            bulk_commit_group();
        }
        item = next;
        cur = nxt;
        rp = np;
    }

    // ---- teardown: a CTA whose bounded wait ran out lets its copies land ------
    tc_fence_before();
    __syncthreads();
    if (fail && pt == 0) {
        atomicAdd(&g_tc_timeouts, 1);
        if (raw_pending) mbar_wait(&bars[0], raw_phase & 1, kWaitLimit, kSuspendNs);
    }
    if (pt == 0) bulk_wait_all();                          // record stores done before the CTA exits
    __syncthreads();
    if (pw == 0) tmem_dealloc(tmem, kPrepTmemCols);
}

// The one-kernel pass (no chunk records): warps 0-3 and 8-11 solve each
// chunk's preparation inline, one chunk ahead of the chain warps 4-7.
__global__ void __launch_bounds__(kThreads, 1)
chunk_tc_kernel(const ChunkParams p, const __grid_constant__ Maps maps) {
    griddep_wait();   // everything the grid before wrote (maps, states, even cu_seqlens)
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float* sA = reinterpret_cast<float*>(sm + kOffA);
    float* sT = reinterpret_cast<float*>(sm + kOffT);
    float* sTmp = reinterpret_cast<float*>(sm + kOffTmp);
    float* vGam = reinterpret_cast<float*>(sm + kOffVec);   // prep: g, then gamma * log2(e)
    float* vEg = vGam + kC;                                 // prep: Gamma
    float* vBeta = vEg + kC;                                // prep: beta
    float* vRk = vBeta + kC;                                // prep: 1/|k_i|
    float* vRq = vRk + kC;                                  // prep: 1/|q_t|
    float* vEnd = vRq + kC;                                 // prep: exp(min(gamma_S - gamma_i, 0)) r_k,i
    float* vFb = vEnd + kC;                                 // prep: beta_i (column factor)
    float* vFbg = vFb + kC;                                 // prep: beta_i Gamma_i r_k,i
    float* vCol = vFbg + kC;                                // prep: gamma_j - log2 r_k,j (log2 domain)
    float* vRowA = vCol + kC;                               // prep: gamma_i + log2 r_k,i
    float* vRowP = vRowA + kC;                              // prep: gamma_t + log2 r_q,t
    float* sG = vRowP + kC;                                 // prep: [2][64] g staging (cp.async)
    float* sB = sG + 2 * kC;                                // prep: [2][64] beta staging
    float* cE = sB + 2 * kC;                                // chain: [2][64] end weights
    float* cGS = cE + 2 * kC;                               // chain: [2] exp(gamma_S)
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kOffBar);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kOffBar + kNumBars * 8);
    volatile int* s_err = reinterpret_cast<volatile int*>(sm + kOffBar + kNumBars * 8 + 4);
    int* s_tma_last = reinterpret_cast<int*>(sm + kOffBar + kNumBars * 8 + 8);   // [2]

    const int h = blockIdx.x, n = seq_of_row(p.cu, p.B, blockIdx.y);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;                 // TMEM lane of this thread
    const uint32_t lane_addr = uint32_t(quarter * 32) << 16;
    // The chain: warps 4-7 (all columns of their TMEM lanes).
    const bool is_chain = warp >= 4 && warp < 8;
    constexpr int hc = 0;
    constexpr int kHalves = 2;
    constexpr uint32_t kChainN = kChainThreads;
    const int kh = h / (p.Hv / p.Hk);
    const int Hv = p.Hv;

    int64_t t_end_all = p.cu[p.B];
    if (t_end_all > p.t_cap) t_end_all = p.t_cap;
    int64_t t0 = p.cu[n], t1 = p.cu[n + 1];
    t0 = t0 < 0 ? 0 : (t0 > t_end_all ? t_end_all : t0);
    t1 = t1 < t0 ? t0 : (t1 > t_end_all ? t_end_all : t1);
    const int seq_chunks = ceil_div32(t1 - t0, p.chunk);
    const size_t sbase = (size_t(n) * Hv + h) * kD * kD;

    // ---- which part of the sequence this CTA runs, and in which mode ------------
    int seg = 0, mode = kModeFull;
    if (p.seg_phase == 1 && blockIdx.z > 0) {
        seg = int(blockIdx.z + 1) / 2;
        mode = (blockIdx.z & 1) ? kModeOffset : kModeTransition;
    }
    // Segments of seg_chunks chunks; when they do not divide the sequence,
    // segment 0 is the short one (the later segments' chunk ranges then
    // depend only on the sequence's chunk count and L).
    int c_begin = 0, c_end = seq_chunks;
    if (p.seg_phase) {
        const int L = p.seg_chunks;
        const int short_by = ((seq_chunks + L - 1) / L) * L - seq_chunks;
        c_begin = seg == 0 ? 0 : seg * L - short_by;
        c_end = min((seg + 1) * L - short_by, seq_chunks);
    }
    if (c_begin >= c_end && !(seg == 0 && mode == kModeFull)) return;   // no such segment
    const int nchunks = c_end > c_begin ? c_end - c_begin : 0;
    const int64_t seq_t0 = t0;
    t0 += int64_t(c_begin) * p.chunk;                   // first token of this CTA's part
    const bool last_seg = c_end >= seq_chunks;
    // Every pass writes its outputs: the full pass the final ones, the offset
    // pass those from a zero incoming state (to the output, completed by
    // seg_out_kernel), the transition pass the output map G.
    float* slot = nullptr;                              // B, M, S of this segment
    float* next_slot = nullptr;                         // of the next segment
    if (p.seg_phase) {
        const int64_t seg_tokens = int64_t(p.seg_chunks) * p.chunk;
        const int64_t sl = seg_slot32(seq_t0, n, seg, seg_tokens);
        slot = p.seg_ws + (size_t(h) * p.seg_slots + sl) * 3 * kD * kD;
        next_slot = slot + 3 * kD * kD;
    }
    // incoming state: state_in (segment 0), zero (offset pass) or the identity
    // (transition pass)
    const float* init_src = seg == 0 && p.state_in ? p.state_in + sbase : nullptr;
    const bool init_identity = mode == kModeTransition;
    // final state: state_out (last segment), S_1 (segment 0 of phase 1), B_s / M_s
    // (fp32, [dk][dv]) or, for S_1 and M_s, the bf16 hi / lo images that
    // seg_out_kernel copies straight into shared memory: S_1^T K-major (row =
    // value column) and M_s^T MN-major (row = key row of the input side), in
    // both cases row = this thread's TMEM lane, 128-byte swizzled.
    float* final_dst = nullptr;
    uint8_t* img_dst = nullptr;
    if (mode == kModeFull) {
        if (last_seg) final_dst = p.state_out ? p.state_out + sbase : nullptr;
        else if (p.seg_phase == 1) img_dst = reinterpret_cast<uint8_t*>(next_slot + 2 * kD * kD);
    } else if (mode == kModeOffset) {
        final_dst = slot;
    } else {
        img_dst = reinterpret_cast<uint8_t*>(slot + kD * kD);
    }

    if (tid == 0) {
        for (int i = 0; i < int(kNumBars); ++i) mbar_init(&bars[i], 1);
        fence_mbar_init();
        *s_err = 0;
        s_tma_last[0] = s_tma_last[1] = -1;
        tma_prefetch_desc(&maps.q);
        tma_prefetch_desc(&maps.k);
        tma_prefetch_desc(&maps.v);
    }
    __syncwarp();
    if (warp == 0) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tZ = tmem + kColZ, tZb = tmem + kColZb, tX = tmem + kColX, tO = tmem + kColO,
                   tGW = tmem + kColGW, tU = tmem + kColU;

    auto stage_ptr = [&](int c) { return sm + uint32_t(c & 1) * kStageBytes; };
    auto chunk_start = [&](int c) { return t0 + int64_t(c) * p.chunk; };
    auto tma_ok = [&](int c) { return chunk_start(c) + kC <= t_end_all; };
    auto issue_tma = [&](int c) {
        uint8_t* kq = stage_ptr(c);
        uint8_t* vv = kq + kStageKQ;
        uint64_t* bar = &bars[B_RAW0 + (c & 1)];
        const int y = int(chunk_start(c));
        s_tma_last[c & 1] = c;
        mbar_arrive_expect_tx(bar, kStageBytes);
        tma_load_2d(kq + 0, &maps.k, bar, kh * kD, y);
        tma_load_2d(kq + 16384, &maps.k, bar, kh * kD + 64, y);
        tma_load_2d(kq + 8192, &maps.q, bar, kh * kD, y);
        tma_load_2d(kq + 24576, &maps.q, bar, kh * kD + 64, y);
        tma_load_2d(vv + 0, &maps.v, bar, h * kD, y);
        tma_load_2d(vv + 8192, &maps.v, bar, h * kD + 64, y);
    };
    // A failed (timed-out) wait marks this thread; each group votes at its
    // barriers (named_sync_or) and leaves its loop together.
    auto wait = [&](int slot, uint32_t parity) { return mbar_wait(&bars[slot], parity, kWaitLimit, kSuspendNs); };

    if (tid == 0) {
        if (nchunks > 0 && tma_ok(0)) issue_tma(0);
        if (nchunks > 1 && tma_ok(1)) issue_tma(1);
    }
    __syncwarp();

    if (!is_chain) {
        // ================================================================ prep
        // Thread 0 alone polls mbarriers; the group learns the outcome through
        // a voting named barrier (many pollers would starve the other warps).
        const int pt = tid < 128 ? tid : tid - 128;      // 0..255
        const int pw = pt >> 5;                          // prep warp 0..7
        const int phalf = tid >= 256 ? 1 : 0;            // column half of TMEM reads
        const __nv_bfloat16* gq = static_cast<const __nv_bfloat16*>(p.q);
        const __nv_bfloat16* gk = static_cast<const __nv_bfloat16*>(p.k);
        const __nv_bfloat16* gv = static_cast<const __nv_bfloat16*>(p.v);
        const uint32_t id_gram = idesc_bf16(128, 64, 0, 0);
        const uint32_t id_uw = idesc_bf16(128, 64, 1, 0);   // A MN-major, B K-major
        const uint64_t dTb = smem_desc(smem_u32(sm + kOffTb), 16, 1024, kSwizzle128B);
        // g and beta of chunk c arrive in staging slot c & 1 by cp.async,
        // issued one chunk ahead (rows past the sequence are zero).
        auto stage_gb = [&](int c) {
            if (pt < kC) {
                const int64_t t = chunk_start(c) + pt;
                float* dg = sG + (c & 1) * kC + pt;
                float* db = sB + (c & 1) * kC + pt;
                if (pt < p.chunk && t < t1) {
                    cp_async4(dg, p.g + t * Hv + h);
                    cp_async4(db, p.beta + t * Hv + h);
                } else {
                    *dg = 0.f;
                    *db = 0.f;
                }
            }
            cp_async_commit();
        };
        // T is lower triangular: its upper triangle is zeroed once here and
        // never written again (each chunk writes the diagonal blocks whole
        // and the blocks below them).
        for (int idx = pt; idx < kC * kLdA; idx += kPrepThreads) sT[idx] = 0.f;
        if (nchunks > 0) stage_gb(0);
        bool fail = false;
        for (int c = 0; c < nchunks; ++c) {
            const int b = c & 1;
            uint8_t* kq = stage_ptr(c);
            uint8_t* vv = kq + kStageKQ;
            const int64_t cs = chunk_start(c);
            const int rows = int(t1 - cs < p.chunk ? t1 - cs : p.chunk);
            // ---- g, beta of this chunk (staged); stage the next chunk's ----------
            cp_async_wait_all();
            named_sync(kBarPrep, kPrepThreads);
            if (pt < kC) {
                vGam[pt] = sG[b * kC + pt];
                vBeta[pt] = sB[b * kC + pt];
            }
            if (c + 1 < nchunks) stage_gb(c + 1);
            // ---- raw tiles ----------------------------------------------------
            bool lf = false;
            if (tma_ok(c)) {
                if (tid == 0) lf = !wait(B_RAW0 + b, uint32_t((c >> 1) & 1));
            } else {
                if (tid == 0 && c >= 2) lf = !wait(B_SFREE0 + b, uint32_t(((c - 2) >> 1) & 1));
                __syncwarp();
                if (named_sync_or(kBarPrep, kPrepThreads, lf)) { fail = true; break; }
                for (int idx = pt; idx < kC * 16; idx += kPrepThreads) {
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
                fence_proxy_async_smem();
            }
            __syncwarp();
            tc_fence_before();
            if (named_sync_or(kBarPrep, kPrepThreads, lf)) { fail = true; break; }
            tc_fence_after();
            // ---- Gram MMA; cumsum (log2 domain); row norms ----------------------
            if (tid == 32) {
                const uint64_t d0 = smem_desc(smem_u32(kq), 16, 1024, kSwizzle128B);
#pragma unroll
                for (int s = 0; s < 8; ++s) {
                    const uint32_t off = uint32_t(s >> 2) * 16384u + uint32_t(s & 3) * 32u;
                    umma_f16(tGW, d0 + (off >> 4), d0 + (off >> 4), id_gram, s > 0);
                }
                umma_commit(&bars[B_GRAM]);
            }
            __syncwarp();
            if (pw == 0) {
                float a = vGam[2 * lane], bb = vGam[2 * lane + 1];
                bb += a;
                float s = bb;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const float u = __shfl_up_sync(0xffffffffu, s, o);
                    if (lane >= o) s += u;
                }
                a += s - bb;
                vGam[2 * lane] = a * kLog2e;                   // gamma * log2(e)
                vGam[2 * lane + 1] = s * kLog2e;
            }
            {
                // 128 rows (K 0..63, Q 0..63); two threads per row, 64 columns each
                const int r = pt >> 1, part = pt & 1;
                const int isq = r >= kC, tr = r & 63;
                const uint8_t* base = kq + (isq ? 8192 : 0);
                float ss = 0.f;
#pragma unroll
                for (int m = 0; m < 8; ++m) {
                    float v[8];
                    load_chunk8(base + toff(tr, part * 64 + m * 8, 16384), v);
#pragma unroll
                    for (int q = 0; q < 8; ++q) ss = fmaf(v[q], v[q], ss);
                }
                ss += __shfl_xor_sync(0xffffffffu, ss, 1);
                if (part == 0) (isq ? vRq : vRk)[tr] = p.l2norm ? rsqrtf(ss + p.eps) : 1.f;
            }
            named_sync(kBarPrep, kPrepThreads);
            if (pt < kC) {
                const float gm = vGam[pt];
                const float eg = exp2f(gm);
                vEg[pt] = eg;
                vEnd[pt] = pt < rows ? exp2f(fminf(vGam[rows - 1] - gm, 0.f)) * vRk[pt] : 0.f;
                vFb[pt] = vBeta[pt];
                vFbg[pt] = vBeta[pt] * eg * vRk[pt];
                const float lk = log2f(vRk[pt]);           // the masks' 2^(row_i - col_j)
                vCol[pt] = gm - lk;
                vRowA[pt] = gm + lk;
                vRowP[pt] = gm + log2f(vRq[pt]);
            }
            // ---- masks and decays on the Gram matrices --------------------------
            if (tid == 0) {
                if (c >= 2) lf = !wait(B_PFREE0 + b, uint32_t(((c - 2) >> 1) & 1));
                lf = lf || !wait(B_GRAM, uint32_t(c & 1));
            }
            __syncwarp();
            if (named_sync_or(kBarPrep, kPrepThreads, lf)) { fail = true; break; }
            tc_fence_after();
            if (phalf == 1 && (pw & 1) == 0) {
                // prep warps 4 and 6: rows 0-31 of A and of P against columns
                // 32-63, every entry masked (j > i, j > t)
                const int r0 = row & (kC - 1);
                if (row < kC) {
#pragma unroll
                    for (int q = 0; q < 32; q += 4)
                        *reinterpret_cast<float4*>(sA + r0 * kLdA + 32 + q) = make_float4(0.f, 0.f, 0.f, 0.f);
                } else {
                    uint8_t* phi = sm + kOffP + uint32_t(b * 2) * 8192u;
                    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                    for (int q = 0; q < 32; q += 8) {
                        const uint32_t o = toff(r0, 32 + q, 8192);
                        *reinterpret_cast<uint4*>(phi + o) = z;
                        *reinterpret_cast<uint4*>(phi + 8192 + o) = z;
                    }
                }
            } else {
                float v[32];
                tmem_ld32(tGW + lane_addr + phalf * 32, v);
                // A_ij = beta_i 2^(row_i - col_j) k_i.k_j (j < i), P_tj =
                // 2^(row_t - col_j) q_t.k_j (j <= t): decays and row norms in
                // one power of two (g <= 0: the exponents need no clamp)
                if (row < kC) {
                    const int i = row;
                    const float bi = vBeta[i], ai = vRowA[i];
#pragma unroll
                    for (int q = 0; q < 32; q += 4) {
                        const float4 c4 = *reinterpret_cast<const float4*>(vCol + phalf * 32 + q);
                        const float cj[4] = {c4.x, c4.y, c4.z, c4.w};
                        float a4[4];
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const int j = phalf * 32 + q + u;
                            a4[u] = (i < rows && j < i) ? bi * (v[q + u] * fast_exp2(ai - cj[u])) : 0.f;
                        }
                        // 16-byte stores: with the 68-float row stride the 8 lanes of
                        // each store phase hit disjoint banks
                        *reinterpret_cast<float4*>(sA + i * kLdA + phalf * 32 + q) = make_float4(a4[0], a4[1], a4[2], a4[3]);
                    }
                } else {
                    const int t = row - kC;
                    const float at = vRowP[t];
#pragma unroll
                    for (int q = 0; q < 32; q += 4) {
                        const float4 c4 = *reinterpret_cast<const float4*>(vCol + phalf * 32 + q);
                        const float cj[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const int j = phalf * 32 + q + u;
                            v[q + u] = (t < rows && j <= t) ? v[q + u] * fast_exp2(at - cj[u]) : 0.f;
                        }
                    }
                    uint8_t* phi = sm + kOffP + uint32_t(b * 2) * 8192u;
#pragma unroll
                    for (int q = 0; q < 32; q += 8) {
                        const uint32_t o = toff(t, phalf * 32 + q, 8192);
                        store_split8(phi + o, phi + 8192 + o, v + q);
                    }
                }
            }
            named_sync(kBarPrep, kPrepThreads);
            // ---- blocked inverse; T diag(beta), T diag(beta Gamma r_k) as hi + lo -
            block_inverse_64(sA, sT, sTmp, pt);
            // a prep warp takes 32 rows of one 8-column group; the groups above
            // the diagonal are zeros, written without the arithmetic
            for (int idx = pt; idx < kC * 8; idx += kPrepThreads) {
                const int t = idx & (kC - 1), i0 = (idx >> 6) * 8;
                const uint32_t o = toff(t, i0, 8192);
                if (i0 > (t | 31)) {
                    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
                    *reinterpret_cast<uint4*>(sm + kOffTb + o) = z;
                    *reinterpret_cast<uint4*>(sm + kOffTb + 8192 + o) = z;
                    *reinterpret_cast<uint4*>(sm + kOffTb + 16384 + o) = z;
                    *reinterpret_cast<uint4*>(sm + kOffTb + 24576 + o) = z;
                    continue;
                }
                float a[8], bg[8], fb[8], fbg[8];
                *reinterpret_cast<float4*>(fb) = *reinterpret_cast<const float4*>(vFb + i0);
                *reinterpret_cast<float4*>(fb + 4) = *reinterpret_cast<const float4*>(vFb + i0 + 4);
                *reinterpret_cast<float4*>(fbg) = *reinterpret_cast<const float4*>(vFbg + i0);
                *reinterpret_cast<float4*>(fbg + 4) = *reinterpret_cast<const float4*>(vFbg + i0 + 4);
                float tr[8];
                *reinterpret_cast<float4*>(tr) = *reinterpret_cast<const float4*>(sT + t * kLdA + i0);
                *reinterpret_cast<float4*>(tr + 4) = *reinterpret_cast<const float4*>(sT + t * kLdA + i0 + 4);
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    a[q] = tr[q] * fb[q];
                    bg[q] = tr[q] * fbg[q];
                }
                store_split8(sm + kOffTb + o, sm + kOffTb + 8192 + o, a);
                store_split8(sm + kOffTb + 16384 + o, sm + kOffTb + 24576 + o, bg);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            named_sync(kBarPrep, kPrepThreads);
            if (tid == 0) {
                if (c > 0) lf = !wait(B_XREAD, uint32_t((c - 1) & 1));
                if (!lf) {
                    tc_fence_after();
                    const uint64_t dV = smem_desc(smem_u32(vv), 8192, 1024, kSwizzle128B);
                    const uint64_t dK = smem_desc(smem_u32(kq), 16384, 1024, kSwizzle128B);
#pragma unroll
                    for (int part = 0; part < 2; ++part)
#pragma unroll
                        for (int s = 0; s < 4; ++s) {
                            // U0^T = V^T Tb^T (V = 0 in the transition pass) ;  W^T = K^T Tbg^T
                            if (mode != kModeTransition)
                                umma_f16(tX, dV + uint64_t(s * 2048 >> 4),
                                         dTb + uint64_t((part * 8192 + s * 32) >> 4), id_uw, part > 0 || s > 0);
                            umma_f16(tGW, dK + uint64_t(s * 2048 >> 4),
                                     dTb + uint64_t((16384 + part * 8192 + s * 32) >> 4), id_uw, part > 0 || s > 0);
                        }
                    umma_commit(&bars[B_W]);
                }
            }
            // ---- while U0/W run: scaled Q rows in place; chain scalars ----------
            for (int idx = pt; idx < kC * 16; idx += kPrepThreads) {
                const int r = idx >> 4, cc = (idx & 15) * 8;
                uint8_t* ptr = kq + 8192 + toff(r, cc, 16384);
                const float f = r < rows ? vEg[r] * vRq[r] : 0.f;
                float v[8];
                load_chunk8(ptr, v);
#pragma unroll
                for (int q = 0; q < 8; ++q) v[q] *= f;
                store_chunk8(ptr, v);
            }
            if (pt < kC) cE[b * kC + pt] = vEnd[pt];
            if (pt == 0) cGS[b] = vEg[rows - 1];
            if (tid == 0 && !lf) {
                lf = !wait(B_W, uint32_t(c & 1));
                if (c >= 1) lf = lf || !wait(B_WTFREE, uint32_t((c - 1) & 1));
            }
            // ---- -W^T to shared ------------------------------------------------
            if (named_sync_or(kBarPrep, kPrepThreads, lf)) { fail = true; break; }
            tc_fence_after();
            {
                float v[32];
                tmem_ld32(tGW + lane_addr + phalf * 32, v);
#pragma unroll
                for (int q = 0; q < 32; ++q) v[q] = -v[q];
#pragma unroll
                for (int q = 0; q < 32; q += 8)
                    store_chunk8(sm + kOffWt + toff(row, phalf * 32 + q, 16384), v + q);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            named_sync(kBarPrep, kPrepThreads);
            if (tid == 0) mbar_arrive(&bars[B_READY0 + b]);
            __syncwarp();
        }
        if (fail) *s_err = 1;
    } else {
        // ================================================================ chain
        // Thread 128 polls the mbarriers and issues the chain MMAs; the group
        // follows through voting named barriers.
        const int ct = tid - 128;                        // == row
        const bool lead = ct == 0;
        __nv_bfloat16* gout = static_cast<__nv_bfloat16*>(mode == kModeTransition ? p.g_out : p.out);
        const uint32_t id_x = idesc_bf16(128, 64, 0, 1);    // B = -W^T, MN-major
        const uint32_t id_o = idesc_bf16(128, 64, 0, 0);    // B = Qs or P, K-major
        const uint32_t id_z = idesc_bf16(128, 128, 0, 1);   // B = raw K, MN-major [i][d]
        bool fail = false;
        // output rows of the previous chunk, kept as bf16 pairs until the next
        // chunk's MMAs are in flight
        uint32_t opk[32];
        int64_t o_cs = 0;
        int o_rows = 0;
        if (nchunks == 0) {
            if (final_dst)
                for (int d = hc * 64; d < (hc + kHalves) * 64; ++d)
                    final_dst[size_t(d) * kD + row] = init_src ? init_src[size_t(d) * kD + row] : 0.f;
        } else {
            // ---- incoming state: Zb = bf16(Z), Z <- exp(gamma_S(0)) Z -----------
            bool lf = lead && !wait(B_READY0, 0);
            __syncwarp();
            fail = named_sync_or(kBarChain, kChainN, lf);
            const float gs0 = cGS[0];
            for (int hf = 0; hf < 2; ++hf) {
                float z[64];
#pragma unroll
                for (int i = 0; i < 64; ++i) {
                    const int d = hf * 64 + i;
                    z[i] = init_src ? init_src[size_t(d) * kD + row] : (init_identity && d == row ? 1.f : 0.f);
                }
                uint32_t zb[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) zb[i] = pack_bf16x2(z[2 * i], z[2 * i + 1]);
                GDN_TMEM_ST_X16(tZb + lane_addr + hf * 32, zb);
                GDN_TMEM_ST_X16(tZb + lane_addr + hf * 32 + 16, (zb + 16));
#pragma unroll
                for (int i = 0; i < 64; ++i) z[i] *= gs0;
                tmem_st16(tZ + lane_addr + hf * 64, z);
                tmem_st16(tZ + lane_addr + hf * 64 + 16, z + 16);
                tmem_st16(tZ + lane_addr + hf * 64 + 32, z + 32);
                tmem_st16(tZ + lane_addr + hf * 64 + 48, z + 48);
            }
            tmem_st_wait();
            tc_fence_before();
            named_sync(kBarChain, kChainN);
        }
        for (int c = 0; c < nchunks && !fail; ++c) {
            const int b = c & 1;
            uint8_t* kq = stage_ptr(c);
            const int64_t cs = chunk_start(c);
            const int rows = int(t1 - cs < p.chunk ? t1 - cs : p.chunk);
            // ---- U^T = U0^T - Zb W^T ;  O^T = Zb Qs^T --------------------------
            bool lf = false;
            if (lead) {
                lf = !wait(B_READY0 + b, uint32_t((c >> 1) & 1));
                if (!lf) {
                    tc_fence_after();
                    const uint64_t dWt = smem_desc(smem_u32(sm + kOffWt), 16384, 1024,
                                                   kSwizzle128B);
#pragma unroll
                    for (int s = 0; s < 8; ++s)
                        umma_f16_tmemA(tX, tZb + s * 8, dWt + uint64_t(s * 2048 >> 4), id_x,
                                       mode != kModeTransition || s > 0);
                    umma_commit(&bars[B_X]);
                    {
                        const uint64_t dQ = smem_desc(smem_u32(kq + 8192), 16, 1024, kSwizzle128B);
#pragma unroll
                        for (int s = 0; s < 8; ++s) {
                            const uint32_t off = uint32_t(s >> 2) * 16384u + uint32_t(s & 3) * 32u;
                            umma_f16_tmemA(tO, tZb + s * 8, dQ + (off >> 4), id_o, s > 0);
                        }
                    }
                }
            }
            __syncwarp();
            // previous chunk's output rows, while the MMAs run (with records:
            // its O^T, once complete, is staged here and written after the
            // next barrier; its P buffer is free then)
            if (c > 0) {
                __nv_bfloat16* dst = gout + (o_cs * Hv + h) * kD + row;
#pragma unroll
                for (int k = 0; k < kHalves * 16; ++k) {
                    const int i = hc * 16 + k;          // rows 2i, 2i + 1 of the chunk
                    const __nv_bfloat162 pr = *reinterpret_cast<const __nv_bfloat162*>(&opk[k]);
                    if (2 * i < o_rows) dst[int64_t(2 * i) * Hv * kD] = pr.x;
                    if (2 * i + 1 < o_rows) dst[int64_t(2 * i + 1) * Hv * kD] = pr.y;
                }
            }
            if (lead && !lf) lf = !wait(B_X, uint32_t(c & 1));
            __syncwarp();
            if (named_sync_or(kBarChain, kChainN, lf)) { fail = true; break; }
            tc_fence_after();
            if (lead) mbar_arrive(&bars[B_WTFREE]);
            __syncwarp();
            // ---- U (hi, lo) and Us = U diag(e) (hi, lo) into TMEM --------------
            for (int hf = hc; hf < hc + kHalves; ++hf) {
                float x[32];
                tmem_ld32(tX + lane_addr + hf * 32, x);
                const float* e = cE + b * kC + hf * 32;
                uint32_t uh[16], ul[16], sh[16], sl[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const float a0 = x[2 * i], a1 = x[2 * i + 1];
                    split_pair(a0, a1, uh[i], ul[i]);
                    split_pair(a0 * e[2 * i], a1 * e[2 * i + 1], sh[i], sl[i]);
                }
                GDN_TMEM_ST_X16(tU + lane_addr + 0 + hf * 16, uh);
                GDN_TMEM_ST_X16(tU + lane_addr + 32 + hf * 16, ul);
                GDN_TMEM_ST_X16(tU + lane_addr + 64 + hf * 16, sh);
                GDN_TMEM_ST_X16(tU + lane_addr + 96 + hf * 16, sl);
            }
            tmem_st_wait();
            tc_fence_before();
            named_sync(kBarChain, kChainN);
            if (lead) {
                mbar_arrive(&bars[B_XREAD]);
                tc_fence_after();
                const uint64_t dK = smem_desc(smem_u32(kq), 16384, 1024, kSwizzle128B);
                const uint64_t dP = smem_desc(smem_u32(sm + kOffP + uint32_t(b * 2) * 8192u), 16, 1024,
                                              kSwizzle128B);
#pragma unroll
                for (int part = 0; part < 2; ++part)
#pragma unroll
                    for (int s = 0; s < 4; ++s)
                        umma_f16_tmemA(tZ, tU + 64 + part * 32 + s * 8, dK + uint64_t(s * 2048 >> 4), id_z, 1);
                umma_commit(&bars[B_Z]);
                {
                    // (U hi, P hi), (U hi, P lo), (U lo, P hi)
#pragma unroll
                    for (int pr = 0; pr < 3; ++pr)
#pragma unroll
                        for (int s = 0; s < 4; ++s)
                            umma_f16_tmemA(tO, tU + (pr == 2 ? 32 : 0) + s * 8,
                                           dP + uint64_t(((pr == 1 ? 8192 : 0) + s * 32) >> 4), id_o, 1);
                    umma_commit(&bars[B_O]);
                }
            }
            __syncwarp();
            // ---- new state: Zb = bf16(Z); Z <- exp(gamma_S(c+1)) Z --------------
            const bool has_next = c + 1 < nchunks;
            if (lead) {
                lf = !wait(B_Z, uint32_t(c & 1));
                // the O issuer's Zb Qs^T must be done before Zb and the stage are reused
                if (!lf) {
                    mbar_arrive(&bars[B_SFREE0 + b]);
                    if (c + 2 < nchunks && tma_ok(c + 2)) issue_tma(c + 2);
                    if (has_next) lf = !wait(B_READY0 + (b ^ 1), uint32_t(((c + 1) >> 1) & 1));
                }
            }
            __syncwarp();
            if (named_sync_or(kBarChain, kChainN, lf)) { fail = true; break; }
            tc_fence_after();
            const float gsn = has_next ? cGS[b ^ 1] : 1.f;
            for (int hf = hc; hf < hc + kHalves; ++hf) {
                float z[64];
                tmem_ld64(tZ + lane_addr + hf * 64, z);
                uint32_t zb[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) zb[i] = pack_bf16x2(z[2 * i], z[2 * i + 1]);
                GDN_TMEM_ST_X16(tZb + lane_addr + hf * 32, zb);
                GDN_TMEM_ST_X16(tZb + lane_addr + hf * 32 + 16, (zb + 16));
                if (has_next) {
#pragma unroll
                    for (int i = 0; i < 64; ++i) z[i] *= gsn;
                    tmem_st16(tZ + lane_addr + hf * 64, z);
                    tmem_st16(tZ + lane_addr + hf * 64 + 16, z + 16);
                    tmem_st16(tZ + lane_addr + hf * 64 + 32, z + 32);
                    tmem_st16(tZ + lane_addr + hf * 64 + 48, z + 48);
                } else if (img_dst) {
                    // this thread's lane is one row of either image
#pragma unroll
                    for (int i = 0; i < 64; i += 8)
                        store_split8(img_dst + toff(row, hf * 64 + i, 16384),
                                     img_dst + 32768 + toff(row, hf * 64 + i, 16384), z + i);
                } else if (final_dst) {
#pragma unroll
                    for (int i = 0; i < 64; ++i) final_dst[size_t(hf * 64 + i) * kD + row] = z[i];
                }
            }
            tmem_st_wait();
            // ---- output rows to registers (stored during the next chunk) --------
            {
                if (lead) lf = !wait(B_O, uint32_t(c & 1));
                __syncwarp();
                if (named_sync_or(kBarChain, kChainN, lf)) { fail = true; break; }
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < kHalves; ++k) {
                    const int hf = hc + k;
                    float o[32];
                    tmem_ld32(tO + lane_addr + hf * 32, o);
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        opk[k * 16 + i] = pack_bf16x2(o[2 * i] * p.q_scale, o[2 * i + 1] * p.q_scale);
                }
            }
            o_cs = cs;
            o_rows = rows;
            tc_fence_before();
            named_sync(kBarChain, kChainN);
            if (lead) mbar_arrive(&bars[B_PFREE0 + b]);
            __syncwarp();
        }
        if (!fail && nchunks > 0) {
            __nv_bfloat16* dst = gout + (o_cs * Hv + h) * kD + row;
#pragma unroll
            for (int k = 0; k < kHalves * 16; ++k) {
                const int i = hc * 16 + k;
                const __nv_bfloat162 pr = *reinterpret_cast<const __nv_bfloat162*>(&opk[k]);
                if (2 * i < o_rows) dst[int64_t(2 * i) * Hv * kD] = pr.x;
                if (2 * i + 1 < o_rows) dst[int64_t(2 * i + 1) * Hv * kD] = pr.y;
            }
        }
        if (fail) *s_err = 1;
    }

    // ---- teardown -----------------------------------------------------------------
    tc_fence_before();
    __syncthreads();
    if (*s_err && tid == 0) {
        atomicAdd(&g_tc_timeouts, 1);
        // let TMA copies still in flight land before shared memory goes away
        for (int st = 0; st < 2; ++st) {
            const int c = s_tma_last[st];
            if (c >= 0) mbar_wait(&bars[B_RAW0 + st], uint32_t((c >> 1) & 1), kWaitLimit, kSuspendNs);
        }
    }
    __syncwarp();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

// ---- state pass over the chunk records --------------------------------------------
// With the records of chunk_prep_kernel a CTA per (value head, sequence,
// segment pass) carries the transposed state Z = S^T through its chunks.  Per
// chunk c (rows i, value columns j):
//   [X | O] = Zb [-W^T | Qs^T]          one N = 128 product, A = Zb from TMEM
//   U^T = U0^T + X,  Us^T = U^T diag(e)  Us as bf16 hi + lo, U as bf16
//   Z += Us^T K                          Z pre-scaled by exp(gamma_S)
//   O += U^T P^T                         (U, P hi), (U, P lo)
//   Zb = bf16(Z), Z <- exp(gamma_S(c+1)) Z
// Roles.  An MMA issue blocks the issuing thread at the tensor pipe's pace
// (about 70 cycles per instruction), so one thread of a warp of its own (the
// MMA issuer) issues every product, and one thread of another (the copier)
// every record copy (the WQ tile, P and U0^T, K and the vectors of a chunk
// into one of two slots, a chunk ahead) and the output tile stores.  Sixteen
// epilogue warps share every epilogue: four per
// TMEM lane quarter, each a quarter of the columns.  The hand-offs are
// mbarriers: the issuer's commits (X, Z, O done) and one arrival per epilogue
// warp (Us written, U written, output tile staged, Zb written).  The
// dependent chain of a chunk is [X | O] product -> Us epilogue -> Z product ->
// Zb epilogue; U, the state's pre-scaling, the output products and the
// previous chunk's output tile all fill the gaps.  The output products of
// chunk c - 1 are issued right behind chunk c's [X | O] product (U is double
// buffered for them), so they run while the Us epilogue works.
constexpr uint32_t kStEpiWarps = 16;
constexpr uint32_t kStEpiThreads = kStEpiWarps * 32;
constexpr uint32_t kStThreads = kStEpiThreads + 64;       // + the MMA issuer's and the copier's warps
// Shared memory: two slots of [WQ tile (32 KB) | P hi, lo (16 KB) | U0^T fragments
// (32 KB) | K (16 KB)] (P and U0^T as one copy: they follow each other in the
// record), two output staging tiles (16 KB each), the two slots' record
// vectors (512 B each).
constexpr uint32_t kStSlot = 98304;
constexpr uint32_t kStOffP = 32768, kStOffU = 49152, kStOffK = 81920;
static_assert(kStOffP - 0 == kRecP - kRecWQ && kStOffU - kStOffP == kRecU - kRecP, "slot mirrors the record");
constexpr uint32_t kStOffO = 2 * kStSlot;
constexpr uint32_t kStOffVec = kStOffO + 2 * 16384;
constexpr uint32_t kStOffBar = kStOffVec + 2 * 512;
enum : int {
    ST_FULL0 = 0,        // slot b's record copies landed (issuer's expect_tx)
    ST_X = 2,            // [X | O] product of the chunk done
    ST_Z = 3,            // state update done
    ST_O0 = 4,           // output products of a chunk into O buffer b done (and every earlier product)
    ST_UREADY = 6,       // Us in TMEM (one arrival per epilogue warp)
    ST_ZBREADY = 7,      // Zb in TMEM
    ST_OSTAGED = 8,      // output tile staged
    ST_SFREE0 = 9,       // staging tile b read by its store
    ST_UHREADY = 11,     // U in TMEM
    ST_DRAIN = 12,
    ST_IMG = 13,         // the final state's image staged (one arrival per epilogue warp)
    ST_NBARS = 14
};
constexpr uint32_t kStSmemBytes = kStOffBar + ST_NBARS * 8 + 16 + 1024;
static_assert(kStSmemBytes <= 232448, "dynamic shared memory above the 227 KB per-block limit");
// TMEM: Z (128) | Zb (64) | O odd (64) | X (64) | O even (64) | U even, U odd, Us hi, Us lo (4 x 32).
// [X | O even] and [O odd | X] are the two N = 128 accumulators of the merged product.
constexpr uint32_t kStColZ = 0, kStColZb = 128, kStColOodd = 192, kStColX = 256, kStColOeven = 320,
                   kStColU = 384;

__global__ void __launch_bounds__(kStThreads, 1)
chunk_state_kernel(const ChunkParams p, const __grid_constant__ Maps maps) {
    // Up to the wait below this reads cu_seqlens only: an input of the call,
    // which no kernel writes and which the preparation (always the grid
    // before, itself behind a full wait) has read; so the index arithmetic
    // runs while the preparation's last CTAs finish.
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kStOffBar);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kStOffBar + ST_NBARS * 8);
    volatile int* s_err = reinterpret_cast<volatile int*>(sm + kStOffBar + ST_NBARS * 8 + 4);
    volatile int* s_issued = reinterpret_cast<volatile int*>(sm + kStOffBar + ST_NBARS * 8 + 8);

    const int h = blockIdx.x, n = seq_of_row(p.cu, p.B, blockIdx.y);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool is_issuer = warp == int(kStEpiWarps);
    const bool is_copier = warp == int(kStEpiWarps) + 1;
    const int quarter = warp & 3, sub = (warp >> 2) & 3;
    const int row = quarter * 32 + lane;                 // TMEM lane of this thread (value column j)
    const uint32_t lane_addr = uint32_t(quarter * 32) << 16;
    const int kh = h / (p.Hv / p.Hk);
    const int Hv = p.Hv;

    int64_t t_end_all = p.cu[p.B];
    if (t_end_all > p.t_cap) t_end_all = p.t_cap;
    int64_t t0 = p.cu[n], t1 = p.cu[n + 1];
    t0 = t0 < 0 ? 0 : (t0 > t_end_all ? t_end_all : t0);
    t1 = t1 < t0 ? t0 : (t1 > t_end_all ? t_end_all : t1);
    const int seq_chunks = ceil_div32(t1 - t0, p.chunk);
    const size_t sbase = (size_t(n) * Hv + h) * kD * kD;
    int seg = 0, mode = kModeFull;
    if (p.seg_phase == 1 && blockIdx.z > 0) {
        seg = int(blockIdx.z + 1) / 2;
        mode = (blockIdx.z & 1) ? kModeOffset : kModeTransition;
    }
    // Segments of seg_chunks chunks; segment 0 is the short one when they do
    // not divide the sequence.
    int c_begin = 0, c_end = seq_chunks;
    if (p.seg_phase) {
        const int L = p.seg_chunks;
        const int short_by = ((seq_chunks + L - 1) / L) * L - seq_chunks;
        c_begin = seg == 0 ? 0 : seg * L - short_by;
        c_end = min((seg + 1) * L - short_by, seq_chunks);
    }
    if (c_begin >= c_end && !(seg == 0 && mode == kModeFull)) return;   // no such segment
    const int nchunks = c_end > c_begin ? c_end - c_begin : 0;
    const int64_t slot0 = int64_t(uint32_t(t0) / uint32_t(p.chunk)) + n + c_begin;   // record slot of this CTA's first chunk
    const int64_t seq_t0 = t0;
    t0 += int64_t(c_begin) * p.chunk;
    const bool last_seg = c_end >= seq_chunks;
    const CUtensorMap* omap = mode == kModeTransition ? &maps.g : &maps.o;
    float* slot = nullptr;
    float* next_slot = nullptr;
    if (p.seg_phase) {
        const int64_t seg_tokens = int64_t(p.seg_chunks) * p.chunk;
        const int64_t sl = seg_slot32(seq_t0, n, seg, seg_tokens);
        slot = p.seg_ws + (size_t(h) * p.seg_slots + sl) * 3 * kD * kD;
        next_slot = slot + 3 * kD * kD;
    }
    // incoming state: state_in (segment 0), zero (offset pass) or the identity
    // (transition pass); final state: state_out (last segment), the S_1 image
    // (segment 0 of phase 1), B_s (fp32) or the M_s^T image
    const float* init_src = seg == 0 && p.state_in ? p.state_in + sbase : nullptr;
    const bool init_identity = mode == kModeTransition;
    const bool has_u0 = mode != kModeTransition;
    float* final_dst = nullptr;
    uint8_t* img_dst = nullptr;
    if (mode == kModeFull) {
        if (last_seg) final_dst = p.state_out ? p.state_out + sbase : nullptr;
        else if (p.seg_phase == 1) img_dst = reinterpret_cast<uint8_t*>(next_slot + 2 * kD * kD);
    } else if (mode == kModeOffset) {
        final_dst = slot;
    } else {
        img_dst = reinterpret_cast<uint8_t*>(slot + kD * kD);
    }
    auto record = [&](int c) {
        return p.prep_ws + (size_t(h) * size_t(p.prep_slots) + size_t(slot0 + c)) * kPrepRecordBytes;
    };
    auto chunk_start = [&](int c) { return t0 + int64_t(c) * p.chunk; };
    auto chunk_rows = [&](int c) {
        const int64_t cs = chunk_start(c);
        return int(t1 - cs < p.chunk ? t1 - cs : p.chunk);
    };
    // A chunk's output tile goes out by TMA when every row of the box is this
    // sequence's or lies past the buffers; else as 16-byte rows (the box's
    // other rows belong to the next sequence).
    auto tile_by_tma = [&](int c) { return chunk_rows(c) == kC || chunk_start(c) + chunk_rows(c) >= p.t_cap; };
    auto wait = [&](int b, uint32_t parity) { return mbar_wait(&bars[b], parity, kWaitLimit, kSuspendNs); };
    // the hand-offs of the chunk chain: polled (see mbar_spin)
    auto spin = [&](int b, uint32_t parity) { return mbar_spin(&bars[b], parity, kWaitLimit); };

    // The record operands of chunk c into slot c & 1: the merged B
    // tile (the record's WQ tile, whose order matches the accumulator
    // pair [X | O even] or [O odd | X] of the chunk's parity), P hi | lo
    // with U0^T, the raw K tile (rows at or past the buffers' end read
    // as zero; rows past the sequences' end are cleared by the
    // epilogue warps) and the vectors.
    auto issue_copies = [&](int c) {
        const int b = c & 1;
        uint8_t* sp = sm + uint32_t(b) * kStSlot;
        const uint8_t* rec = record(c);
        uint64_t* bar = &bars[ST_FULL0 + b];
        mbar_arrive_expect_tx(bar, 32768u + 16384u + 16384u + 512u + (has_u0 ? 32768u : 0u));
        bulk_load(sp, rec + kRecWQ, 32768, bar);
        bulk_load(sp + kStOffP, rec + kRecP, has_u0 ? 49152u : 16384u, bar);
        tma_load_2d(sp + kStOffK, &maps.k, bar, kh * kD, int(chunk_start(c)));
        tma_load_2d(sp + kStOffK + 8192, &maps.k, bar, kh * kD + 64, int(chunk_start(c)));
        bulk_load(sm + kStOffVec + uint32_t(b) * 512u, rec + kRecVec, 512, bar);
        *s_issued = c + 1;
    };
    griddep_wait();   // the records, maps and states the grids before wrote
    // The copier thread sets up the barriers and starts the first record's
    // copies before the block's first barrier.
    if (is_copier && lane == 0) {
        for (int i = 0; i < ST_NBARS; ++i)
            mbar_init(&bars[i], (i == ST_UREADY || i == ST_UHREADY || i == ST_ZBREADY || i == ST_OSTAGED ||
                                 i == ST_IMG)
                                    ? kStEpiWarps : 1);
        fence_mbar_init();
        *s_err = 0;
        *s_issued = 0;
        if (nchunks > 0) {
            tma_prefetch_desc(&maps.k);
            tma_prefetch_desc(omap);
            issue_copies(0);
        }
    }
    __syncwarp();
    if (warp == 0) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tZ = tmem + kStColZ, tZb = tmem + kStColZb, tX = tmem + kStColX, tU = tmem + kStColU;
    auto tO = [&](int c) { return tmem + ((c & 1) ? kStColOodd : kStColOeven); };
    auto tXO = [&](int c) { return tmem + ((c & 1) ? kStColOodd : kStColX); };
    uint8_t* const o_stage = sm + kStOffO;

    if (is_copier) {
        // ============================================================ copier
        if (lane == 0 && nchunks > 0) {
            // the staged output tile of chunk cc to the output (TMA; one bulk
            // group per chunk, empty when the epilogue warps stored the rows);
            // chunk cc - 1's staging tile is free once its store has read it
            auto store_tile = [&](int cc) {
                if (!wait(ST_OSTAGED, uint32_t(cc & 1))) return false;
                const uint8_t* st = o_stage + uint32_t(cc & 1) * 16384u;
                if (tile_by_tma(cc)) {
                    tma_store_2d(omap, st, h * kD, int(chunk_start(cc)));
                    tma_store_2d(omap, st + 8192, h * kD + 64, int(chunk_start(cc)));
                }
                bulk_commit_group();
                bulk_wait_group_read<1>();
                if (cc >= 1) mbar_arrive(&bars[ST_SFREE0 + ((cc - 1) & 1)]);
                return true;
            };
            if (nchunks > 1) issue_copies(1);
            bool fail = false;
            for (int c = 1; c < nchunks && !fail; ++c) {
                // slot (c + 1) & 1 held chunk c - 1, whose products are done once
                // its output products are: it takes chunk c + 1
                if (!wait(ST_O0 + ((c - 1) & 1), uint32_t(((c - 1) >> 1) & 1))) {
                    fail = true;
                    break;
                }
                if (c + 1 < nchunks) issue_copies(c + 1);
                if (!store_tile(c - 1)) fail = true;
            }
            if (!fail && !store_tile(nchunks - 1)) fail = true;
            bulk_wait_all();                              // tile stores done before the CTA exits
            if (fail) *s_err = 1;
        }
    } else if (is_issuer) {
        // ========================================================= MMA issuer
        if (lane == 0 && nchunks > 0) {
            const uint32_t id_xo = idesc_bf16(128, 128, 0, 0);   // B = the merged tile, K-major
            const uint32_t id_o = idesc_bf16(128, 64, 0, 0);     // B = P, K-major
            const uint32_t id_z = idesc_bf16(128, 128, 0, 1);    // B = raw K, MN-major [i][d]
            // O += U^T P^T of chunk cc: (U, P hi), (U, P lo); U of chunk cc in
            // TMEM buffer cc & 1 (written once ST_UHREADY's phase cc completed)
            auto issue_op = [&](int cc) {
                tc_fence_after();
                const uint8_t* sp = sm + uint32_t(cc & 1) * kStSlot;
                const uint64_t dP = smem_desc(smem_u32(sp + kStOffP), 16, 1024, kSwizzle128B);
#pragma unroll
                for (int pr = 0; pr < 2; ++pr)
#pragma unroll
                    for (int s = 0; s < 4; ++s)
                        umma_f16_tmemA(tO(cc), tU + uint32_t(cc & 1) * 32 + s * 8,
                                       dP + uint64_t((pr * 8192 + s * 32) >> 4), id_o, 1);
                umma_commit(&bars[ST_O0 + (cc & 1)]);
            };
            bool fail = false;
            for (int c = 0; c < nchunks && !fail; ++c) {
                const int b = c & 1;
                // ---- [X | O] = Zb [-W^T | Qs^T] ------------------------------------
                // (U of chunk c - 1 is known before this product is issued, so
                // that phase of ST_UHREADY cannot be overtaken)
                if (!spin(ST_FULL0 + b, uint32_t((c >> 1) & 1)) || !spin(ST_ZBREADY, uint32_t(c & 1)) ||
                    (c >= 1 && !spin(ST_UHREADY, uint32_t((c - 1) & 1)))) {
                    fail = true;
                    break;
                }
                tc_fence_after();
                {
                    const uint64_t dB = smem_desc(smem_u32(sm + uint32_t(b) * kStSlot), 16, 1024, kSwizzle128B);
#pragma unroll
                    for (int s = 0; s < 8; ++s) {
                        const uint32_t off = uint32_t(s >> 2) * 16384u + uint32_t(s & 3) * 32u;
                        umma_f16_tmemA(tXO(c), tZb + s * 8, dB + (off >> 4), id_xo, s > 0);
                    }
                    umma_commit(&bars[ST_X]);
                }
                // ---- O += U^T P^T of the previous chunk, behind it -------------------
                if (c >= 1) issue_op(c - 1);
                // ---- Z += Us^T K -------------------------------------------------------
                if (!spin(ST_UREADY, uint32_t(c & 1))) { fail = true; break; }
                tc_fence_after();
                {
                    const uint8_t* sp = sm + uint32_t(b) * kStSlot;
                    const uint64_t dK = smem_desc(smem_u32(sp + kStOffK), 8192, 1024, kSwizzle128B);
#pragma unroll
                    for (int part = 0; part < 2; ++part)
#pragma unroll
                        for (int s = 0; s < 4; ++s)
                            umma_f16_tmemA(tZ, tU + 64 + part * 32 + s * 8, dK + uint64_t(s * 2048 >> 4), id_z, 1);
                    umma_commit(&bars[ST_Z]);
                }
            }
            if (!fail) {
                if (wait(ST_UHREADY, uint32_t((nchunks - 1) & 1))) issue_op(nchunks - 1);
                else fail = true;
            }
            if (fail) *s_err = 1;
        }
    } else {
        // =========================================================== epilogue
        // Thread 0 polls the mbarriers and the sixteen warps follow through a
        // named barrier (every wait below is reached by all of them), so that
        // one thread polls instead of sixteen beside the issuer's polls.
        __nv_bfloat16* gout = static_cast<__nv_bfloat16*>(mode == kModeTransition ? p.g_out : p.out);
        auto warp_wait = [&](int b, uint32_t parity) {
            bool bad = false;
            if (tid == 0) bad = !spin(b, parity);
            return !named_sync_or(kBarPrep, kStEpiThreads, bad);
        };
        auto warp_arrive = [&](int b) {
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[b]);
        };
        // Output tile of chunk cc: O^T read out of TMEM as MMA-ordered
        // fragments (this warp: its 32 lanes, columns 16 sub .. 16 sub + 15)
        // and stored transposed (stmatrix) into staging tile cc & 1 ([64 rows]
        // [128 columns] bf16, 128-byte swizzle); where the tile cannot go out
        // by TMA the warps store its rows.
        auto stage_out = [&](int cc) {
            // staging tile cc & 1 was last read by chunk cc - 2's store
            if (cc >= 2 && !warp_wait(ST_SFREE0 + (cc & 1), uint32_t(((cc - 2) >> 1) & 1))) return false;
            if (!warp_wait(ST_O0 + (cc & 1), uint32_t((cc >> 1) & 1))) return false;
            tc_fence_after();
            uint8_t* st = o_stage + uint32_t(cc & 1) * 16384u;
            uint32_t r[2][8];
            __syncwarp();
#pragma unroll
            for (int u = 0; u < 2; ++u)
                tmem_ld_16x256b_x2(tO(cc) + (uint32_t(quarter * 32 + 16 * u) << 16) + uint32_t(sub * 16), r[u]);
            tmem_ld_wait();
            const int m = lane >> 3, rr = lane & 7;
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                uint32_t f[4];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    f[e] = pack_bf16x2(__uint_as_float(r[u][2 * e]) * p.q_scale,
                                       __uint_as_float(r[u][2 * e + 1]) * p.q_scale);
                const int t = sub * 16 + 8 * (m >> 1) + rr;
                const int j = quarter * 32 + 16 * u + 8 * (m & 1);
                stmatrix_x4_trans(smem_u32(st + toff(t, j, 8192)), f);
            }
            fence_proxy_async_smem();
            if (!tile_by_tma(cc)) {
                // this warp's part of the tile (rows 16 sub .., columns 32 quarter ..)
                __syncwarp();
                const int64_t o_cs = chunk_start(cc);
                const int o_rows = chunk_rows(cc);
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const int idx = lane + 32 * k;
                    const int r2 = sub * 16 + (idx >> 2), col = quarter * 32 + (idx & 3) * 8;
                    if (r2 < o_rows)
                        *reinterpret_cast<uint4*>(gout + ((o_cs + r2) * Hv + h) * kD + col) =
                            *reinterpret_cast<const uint4*>(st + toff(r2, col, 8192));
                }
            }
            tc_fence_before();
            warp_arrive(ST_OSTAGED);
            return true;
        };
        bool fail = false;
        if (nchunks == 0) {
            if (final_dst)
                for (int d = sub * 32; d < sub * 32 + 32; ++d)
                    final_dst[size_t(d) * kD + row] = init_src ? init_src[size_t(d) * kD + row] : 0.f;
        } else {
            {
                // ---- incoming state (this thread: key rows 32 sub .. 32 sub + 31):
                // Zb = bf16(S_0^T), Z = exp(gamma_S(0)) S_0^T
                // (Zb is handed over first: the first product reads it, while Z
                // is read only by the state update, which waits for this warp's
                // Us and with it for these stores)
                const float gs = __ldg(reinterpret_cast<const float*>(record(0) + kRecVec) + kC);
                float z[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int d = sub * 32 + i;
                    z[i] = init_src ? init_src[size_t(d) * kD + row] : (init_identity && d == row ? 1.f : 0.f);
                }
                uint32_t zb[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) zb[i] = pack_bf16x2(z[2 * i], z[2 * i + 1]);
                GDN_TMEM_ST_X16(tZb + lane_addr + sub * 16, zb);
                tmem_st_wait();
                tc_fence_before();
                warp_arrive(ST_ZBREADY);
#pragma unroll
                for (int i = 0; i < 32; ++i) z[i] *= gs;
                tmem_st16(tZ + lane_addr + sub * 32, z);
                tmem_st16(tZ + lane_addr + sub * 32 + 16, z + 16);
            }
            for (int c = 0; c < nchunks; ++c) {
                const int b = c & 1;
                const int64_t cs = chunk_start(c);
                const bool has_next = c + 1 < nchunks;
                // exp(gamma_S) of the next chunk, for the state's pre-scaling
                const float gsn = has_next ? __ldg(reinterpret_cast<const float*>(record(c + 1) + kRecVec) + kC) : 1.f;
                if (!warp_wait(ST_FULL0 + b, uint32_t((c >> 1) & 1)) || !warp_wait(ST_X, uint32_t(c & 1))) {
                    fail = true;
                    break;
                }
                tc_fence_after();
                if (cs + kC > t_end_all) {
                    // K rows past the sequences' end (another caller's rows, or
                    // unset) must not meet the zero rows of Us: clear them
                    uint8_t* kt = sm + uint32_t(b) * kStSlot + kStOffK;
                    const int valid = int(t_end_all - cs);
                    for (int idx = tid; idx < kC * 16; idx += int(kStEpiThreads)) {
                        const int r2 = idx >> 4, cc = (idx & 15) * 8;
                        if (r2 >= valid) *reinterpret_cast<uint4*>(kt + toff(r2, cc, 8192)) = make_uint4(0, 0, 0, 0);
                    }
                    fence_proxy_async_smem();
                }
                // ---- U^T = U0^T + X; Us = U diag(e) as bf16 hi + lo, then U as bf16 ----
                // (this thread: columns 16 sub .. 16 sub + 15 of its lane; U0^T
                // from the slot's copy of the record's fragments, which the
                // preparing thread of that lane and column half wrote as
                // interleaved 16-byte groups)
                {
                    uint32_t xr[16];
                    __syncwarp();
                    GDN_TMEM_LD_X16(tX + lane_addr + sub * 16, xr);
                    const float* ev = reinterpret_cast<const float*>(sm + kStOffVec + uint32_t(b) * 512u) + sub * 16;
                    const float4* us = reinterpret_cast<const float4*>(sm + uint32_t(b) * kStSlot + kStOffU) +
                                       ((quarter + 4 * (sub >> 1)) * 8 + 4 * (sub & 1)) * 32 + lane;
                    float u[16];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const float4 w = has_u0 ? us[k * 32] : make_float4(0.f, 0.f, 0.f, 0.f);
                        u[4 * k] = w.x;
                        u[4 * k + 1] = w.y;
                        u[4 * k + 2] = w.z;
                        u[4 * k + 3] = w.w;
                    }
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 16; ++i) u[i] += __uint_as_float(xr[i]);
                    uint32_t sh[8], sl[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const float2 e2 = *reinterpret_cast<const float2*>(ev + 2 * i);
                        split_pair(u[2 * i] * e2.x, u[2 * i + 1] * e2.y, sh[i], sl[i]);
                    }
                    GDN_TMEM_ST_X8(tU + lane_addr + 64 + sub * 8, sh);
                    GDN_TMEM_ST_X8(tU + lane_addr + 96 + sub * 8, sl);
                    tmem_st_wait();
                    tc_fence_before();
                    warp_arrive(ST_UREADY);
                    uint32_t uh[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) uh[i] = pack_bf16x2(u[2 * i], u[2 * i + 1]);
                    GDN_TMEM_ST_X8(tU + lane_addr + uint32_t(b) * 32 + sub * 8, uh);
                    tmem_st_wait();
                }
                tc_fence_before();
                warp_arrive(ST_UHREADY);
                // ---- the previous chunk's output tile, while the state update runs --
                if (c >= 1 && !stage_out(c - 1)) {
                    fail = true;
                    break;
                }
                // ---- new state: Zb = bf16(Z); Z <- exp(gamma_S(c+1)) Z --------------
                if (!warp_wait(ST_Z, uint32_t(c & 1))) {
                    fail = true;
                    break;
                }
                tc_fence_after();
                {
                    float z[32];
                    tmem_ld32(tZ + lane_addr + sub * 32, z);
                    uint32_t zb[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) zb[i] = pack_bf16x2(z[2 * i], z[2 * i + 1]);
                    GDN_TMEM_ST_X16(tZb + lane_addr + sub * 16, zb);
                    tmem_st_wait();
                    tc_fence_before();
                    warp_arrive(ST_ZBREADY);
                    // the pre-scaling for the next chunk's update (or the final
                    // state) while the next [X | O] product runs
                    if (has_next) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) z[i] *= gsn;
                        tmem_st16(tZ + lane_addr + sub * 32, z);
                        tmem_st16(tZ + lane_addr + sub * 32 + 16, z + 16);
                    } else if (img_dst) {
                        // this thread's lane is one row of either image, staged
                        // in the slot of the (absent) next chunk, whose last
                        // chunk's products are done; then every warp copies a
                        // sixteenth of the staged images out in whole lines
                        uint8_t* st = sm + uint32_t(nchunks & 1) * kStSlot;
#pragma unroll
                        for (int i = 0; i < 32; i += 8)
                            store_split8(st + toff(row, sub * 32 + i, 16384), st + 32768 + toff(row, sub * 32 + i, 16384),
                                         z + i);
                        warp_arrive(ST_IMG);
                        if (!warp_wait(ST_IMG, 0)) {
                            fail = true;
                            break;
                        }
                        const uint4* src = reinterpret_cast<const uint4*>(st) + warp * 256;
                        uint4* dst = reinterpret_cast<uint4*>(img_dst) + warp * 256;
#pragma unroll
                        for (int k = 0; k < 8; ++k) dst[k * 32 + lane] = src[k * 32 + lane];
                    } else if (final_dst) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) final_dst[size_t(sub * 32 + i) * kD + row] = z[i];
                    }
                    tmem_st_wait();
                }
            }
            if (!fail && !stage_out(nchunks - 1)) fail = true;   // the last chunk's output tile
        }
        if (fail) *s_err = 1;
    }

    // ---- teardown ------------------------------------------------------------------
    tc_fence_before();
    __syncthreads();
    if (tid == int(kStEpiThreads)) {
        tc_fence_after();
        // every product the issuer started has completed before TMEM and
        // shared memory go away (a no-op wait on a clean finish)
        umma_commit(&bars[ST_DRAIN]);
        if (!mbar_wait(&bars[ST_DRAIN], 0, kWaitLimit, kSuspendNs)) *s_err = 1;
        if (*s_err) {
            atomicAdd(&g_tc_timeouts, 1);
            // record copies still in flight land before shared memory goes away
            const int issued = *s_issued;
            for (int c = issued - 2 < 0 ? 0 : issued - 2; c < issued; ++c)
                mbar_wait(&bars[ST_FULL0 + (c & 1)], uint32_t((c >> 1) & 1), kWaitLimit, kSuspendNs);
            bulk_wait_all();
        }
    }
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

// ---- segment outputs -----------------------------------------------------------
// Phase 1 leaves, per (value head, sequence): S_1 (the end state of segment
// 0, whose outputs are final), and for every later segment s its offset B_s
// and transition M_s, the outputs O' of its chunks from a zero incoming state
// (in `out`) and its output map G (the outputs from the identity with V = 0,
// in the G buffer).  A chunk's outputs are linear in the segment's incoming
// state, so with S_{s+1} = M_s S_s + B_s every output row is O = O' + G S_s.
//
// seg_out_kernel, grid (Hv, B, output CTAs + final CTA), 320 threads: an
// output CTA takes one chunk group of one segment s >= 1 (ChunkParams::
// seg_gstart; later segments have more groups, as their CTAs first take
// more state steps), forms S_s from S_1 by s - 1 steps and then
// O = O' + G S_s for its chunks.  The final state S_n of the sequence's n
// segments (n - 1 steps) is formed by one more CTA when that fits the wave,
// else by the last group's CTA of segment n - 1 after its outputs.  The CTA
// keeps S^T as bf16 hi and lo images (the A operand: rows = value columns,
// K = key rows); phase 1 leaves S_1 and every M_s^T as such images (M_s^T
// MN-major), which arrive by bulk copy, M double-buffered.  A step is three
// M = N = 128 tcgen05 products, D = S^T M^T from (hi, hi), (hi, lo), (lo, hi),
// then S_{s+1}^T = D + B_s^T in fp32 (TMEM lane = value column) and back to
// images.  An output chunk is one product O^T = bf16(S)^T G^T (the state
// enters output products as a single bf16 in every pass of the scan; B = the
// chunk's G tile, K-major as stored, in a ring of three); O' (a ring of three)
// is added in fp32 in the epilogue, read from its tile in the same fragment
// layout as the result is written back (ldmatrix / stmatrix, transposed), and
// the tile is stored by TMA in place.  During the outputs one thread of an
// issuer warp issues the products (into two TMEM buffers) and the G tile
// loads, one thread of a tile warp the tile stores and the O' tile loads,
// and eight epilogue warps hand over through mbarriers (product done, TMEM
// buffer read, tile written), so that the product of chunk i + 1 and the
// store of chunk i - 1 run while chunk i's epilogue does.
constexpr uint32_t kSoEpiWarps = 8;
constexpr uint32_t kSoEpiThreads = kSoEpiWarps * 32;
constexpr uint32_t kSoThreads = kSoEpiThreads + 64;  // + the issuer's and the tile warp
constexpr int kSoMma = int(kSoEpiThreads);           // the issuer thread
constexpr int kSoCtl = int(kSoEpiThreads) + 32;      // the tile thread
constexpr uint32_t kSoImg = 32768;                  // one 128 x 128 bf16 image, two 16 KB blocks
constexpr uint32_t kSoOffS = 0;                     // S^T hi | lo, K-major
constexpr uint32_t kSoOffM0 = 2 * kSoImg;           // M^T hi | lo, MN-major: buffer 0
constexpr uint32_t kSoOffTile = 4 * kSoImg;         // M^T buffer 1 during the steps, then the tiles
constexpr uint32_t kSoOffM1 = kSoOffTile;
constexpr uint32_t kSoOffG = kSoOffTile;            // G tiles: three of 16 KB
constexpr uint32_t kSoOffP = kSoOffTile + 3 * 16384;   // O' tiles: three of 16 KB
constexpr uint32_t kSoOffBar = kSoOffTile + 6 * 16384;
constexpr uint32_t kSoNumBars = 14;
constexpr uint32_t kSoSmem = kSoOffBar + kSoNumBars * 8 + 16 + 1024;
constexpr uint32_t kSoTmemCols = 256;               // step accumulator (128) | O^T, two buffers of 64
static_assert(kSoOffM1 + 2 * kSoImg <= kSoOffBar, "M^T buffer 1 inside the tile region");
static_assert(kSoSmem <= 232448, "dynamic shared memory above the 227 KB per-block limit");
enum : int {
    SO_STEP = 0,         // the step's products done
    SO_G0 = 1,           // G tile b landed (three)
    SO_P0 = 4,           // O' tile b landed (three)
    SO_O0 = 7,           // output product into TMEM buffer b done (two)
    SO_OFREE0 = 9,       // TMEM buffer b read by the epilogue warps (two; one arrival per warp)
    SO_STAGED0 = 11,     // the result of a chunk written into its tile (two; one arrival per warp)
    SO_DRAIN = 13        // the control thread's products done (teardown after a failure)
};

// This thread's 64 entries of column r = tid % 128 of a row-major 128 x 128
// fp32 matrix, rows (tid / 128) * 64 ... + 63: coalesced across a warp.
__device__ __forceinline__ void so_load_col(const float* src, int tid, float* v) {
    const int r = tid & 127, k0 = (tid >> 7) * 64;
#pragma unroll
    for (int i = 0; i < 64; ++i) v[i] = src[size_t(k0 + i) * kD + r];
}

// Row r = tid % 128, columns (tid / 128) * 64 ... + 63 of a hi / lo image pair.
__device__ __forceinline__ void so_store_row(uint8_t* img, int tid, const float* v) {
    const int r = tid & 127, k0 = (tid >> 7) * 64;
#pragma unroll
    for (int c = 0; c < 64; c += 8) store_split8(img + toff(r, k0 + c, 16384), img + kSoImg + toff(r, k0 + c, 16384), v + c);
}

__global__ void __launch_bounds__(kSoThreads, 1) seg_out_kernel(const ChunkParams p, const __grid_constant__ Maps maps) {
    // Up to the wait below this reads cu_seqlens only (an input of the call,
    // which no kernel writes and which the grids before have read behind
    // their own waits), so the index arithmetic overlaps phase 1's end.
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kSoOffBar);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kSoOffBar + kSoNumBars * 8);
    volatile int* s_err = reinterpret_cast<volatile int*>(sm + kSoOffBar + kSoNumBars * 8 + 4);
    volatile int* s_g_issued = reinterpret_cast<volatile int*>(sm + kSoOffBar + kSoNumBars * 8 + 8);
    volatile int* s_p_issued = reinterpret_cast<volatile int*>(sm + kSoOffBar + kSoNumBars * 8 + 12);
    const int h = blockIdx.x, n = seq_of_row(p.cu, p.B, blockIdx.y), z = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool epi = warp < int(kSoEpiWarps);
    const int Hv = p.Hv;

    int64_t t_end_all = p.cu[p.B];
    if (t_end_all > p.t_cap) t_end_all = p.t_cap;
    int64_t t0 = p.cu[n], t1 = p.cu[n + 1];
    t0 = t0 < 0 ? 0 : (t0 > t_end_all ? t_end_all : t0);
    t1 = t1 < t0 ? t0 : (t1 > t_end_all ? t_end_all : t1);
    const int seq_chunks = ceil_div32(t1 - t0, p.chunk);
    const int L = p.seg_chunks;
    const int nseg = (seq_chunks + L - 1) / L;
    const int short_by = nseg * L - seq_chunks;
    // this CTA's segment s and chunk group g of its segment's groups
    const bool table = p.seg_max - 1 <= kSegTable;
    const int so_ctas = table ? int(p.seg_gstart[p.seg_max - 1]) : (p.seg_max - 1) * p.seg_groups;
    const bool final_role = p.seg_final_cta && z == so_ctas;
    int s = 1, g = 0, groups = 1;                    // steps: s - 1, or nseg - 1 for the final state
    if (final_role) {
        s = nseg - 1;
    } else if (table) {
        while (s < p.seg_max - 1 && z >= int(p.seg_gstart[s])) ++s;
        g = z - int(p.seg_gstart[s - 1]);
        groups = int(p.seg_gstart[s]) - int(p.seg_gstart[s - 1]);
    } else {
        groups = p.seg_groups;
        s = 1 + z / groups;
        g = z % groups;
    }
    if (nseg < 2 || s >= nseg) return;
    if (final_role && p.state_out == nullptr) return;
    int c_lo = 0, c_hi = 0;                          // this CTA's chunks (output role)
    if (!final_role) {
        const int cb = s * L - short_by;
        c_lo = cb + (g * L) / groups;
        c_hi = cb + ((g + 1) * L) / groups;
        if (c_lo >= c_hi) return;
    }
    const int nsteps = final_role ? nseg - 1 : s - 1;
    // the final state after the outputs, by the last group of the last segment
    const bool final_after = !final_role && !p.seg_final_cta && p.state_out != nullptr && s == nseg - 1 &&
                             g == groups - 1;
    const int nout = c_hi - c_lo;
    const bool tiles_early = nsteps < 2;             // M^T buffer 1 (the tile region) never used
    const int64_t seg_tokens = int64_t(L) * p.chunk;
    const float* slots = p.seg_ws + (size_t(h) * p.seg_slots + seg_slot32(t0, n, 0, seg_tokens)) * 3 * kD * kD;
    auto slot_of = [&](int j) { return slots + size_t(j) * 3 * kD * kD; };   // B_j, M_j^T image, S_j image

    griddep_wait();                                  // phase 1's outputs, maps and S_1
    if (tid == 0) {
        for (int i = 0; i < int(kSoNumBars); ++i)
            mbar_init(&bars[i], (i >= SO_OFREE0 && i < SO_DRAIN) ? kSoEpiWarps : 1);
        fence_mbar_init();
        *s_err = 0;
        *s_g_issued = 0;
        *s_p_issued = 0;
    }
    __syncwarp();
    if (warp == 0) {
        tmem_alloc(tmem_slot, kSoTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tD = tmem, tOb = tmem + 128;
    const int quarter = warp & 3, half = (warp >> 2) & 1;
    const int row = quarter * 32 + lane;             // TMEM lane: the value column
    const uint32_t lane_addr = uint32_t(quarter * 32) << 16;
    auto wait = [&](int b, uint32_t parity) { return mbar_wait(&bars[b], parity, kWaitLimit, kSuspendNs); };
    auto chunk_start = [&](int c) { return t0 + int64_t(c) * p.chunk; };
    // Output chunk i's tile goes out by TMA when every row of the box is this
    // sequence's or lies past the buffers; else as 16-byte rows.
    auto out_rows = [&](int i) {
        const int64_t cs = chunk_start(c_lo + i);
        return int(t1 - cs < p.chunk ? t1 - cs : p.chunk);
    };
    auto tile_by_tma = [&](int i) { return out_rows(i) == kC || chunk_start(c_lo + i) + out_rows(i) >= p.t_cap; };
    // The images (64 KB) arrive by cp.async from every thread, one commit
    // group each.  The tile copies are counted, so that a failed CTA can let
    // the ones in flight land before it exits.
    auto load_image = [&](uint8_t* dst, const void* src) {
        const uint8_t* src8 = static_cast<const uint8_t*>(src);
        for (int i = tid; i < int(2 * kSoImg / 16); i += int(kSoThreads)) cp_async16(dst + i * 16, src8 + i * 16);
        cp_async_commit();
    };
    auto load_m = [&](int j, int mb) {               // M_j^T image into buffer mb
        load_image(sm + (mb ? kSoOffM1 : kSoOffM0), slot_of(j) + kD * kD);
    };
    auto issue_g = [&](int i) {                      // G tile of output chunk i
        uint64_t* bar = &bars[SO_G0 + i % 3];
        uint8_t* dst = sm + kSoOffG + uint32_t(i % 3) * 16384u;
        const int y = int(chunk_start(c_lo + i));
        mbar_arrive_expect_tx(bar, 16384);
        tma_load_2d_hint(dst, &maps.g, bar, h * kD, y, l2_evict_first());
        tma_load_2d_hint(dst + 8192, &maps.g, bar, h * kD + 64, y, l2_evict_first());
        *s_g_issued = i + 1;
    };
    auto issue_p = [&](int i) {                      // O' tile of output chunk i
        uint64_t* bar = &bars[SO_P0 + i % 3];
        uint8_t* dst = sm + kSoOffP + uint32_t(i % 3) * 16384u;
        const int y = int(chunk_start(c_lo + i));
        mbar_arrive_expect_tx(bar, 16384);
        tma_load_2d_hint(dst, &maps.o, bar, h * kD, y, l2_evict_first());
        tma_load_2d_hint(dst + 8192, &maps.o, bar, h * kD + 64, y, l2_evict_first());
        *s_p_issued = i + 1;
    };
    // the first G tiles and O' tiles (O' tile i + 2 follows once chunk i is
    // staged, so that the phases of SO_STAGED cannot run two ahead of the
    // tile thread)
    auto issue_tiles = [&]() {
        for (int i = 0; i < nout && i < 3; ++i) issue_g(i);
        for (int i = 0; i < nout && i < 2; ++i) issue_p(i);
    };
    load_image(sm + kSoOffS, slot_of(1) + 2 * kD * kD);  // S_1^T
    if (nsteps > 0 || final_after) load_m(1, 0);
    if (nsteps > 1) load_m(2, 1);
    if (tid == kSoCtl && tiles_early) issue_tiles();
    // the tiles of later chunks toward L2: after the images (a CTA with state
    // steps asks during its last step)
    auto prefetch_tiles = [&](int from, int to) {
        for (int i = from; i < nout && i < to; ++i) {
            const int y = int(chunk_start(c_lo + i));
            tma_prefetch_2d(&maps.g, h * kD, y);
            tma_prefetch_2d(&maps.g, h * kD + 64, y);
            tma_prefetch_2d(&maps.o, h * kD, y);
            tma_prefetch_2d(&maps.o, h * kD + 64, y);
        }
    };
    if (tid == 64 && tiles_early) prefetch_tiles(3, 6);
    __syncwarp();
    bool fail = false;
    const uint64_t dS = smem_desc(smem_u32(sm + kSoOffS), 16, 1024, kSwizzle128B);
    const uint32_t id_step = idesc_bf16(128, 128, 0, 1);      // B = M^T image, MN-major
    // Step j with M_j^T in buffer mb: S_{j+1}^T = S^T M_j^T + B_j^T into the S
    // images, or into state_out; M_{j+2}^T follows into the freed buffer when
    // next_load.  one_more: the copy of M_{j+1} may still be in flight.
    // False when a wait ran out.  (The control warp takes part in the copies
    // and the block barriers only.)
    auto step = [&](int j, int mb, bool to_state, bool next_load, bool one_more) {
        if (one_more)
            cp_async_wait_group<1>();
        else
            cp_async_wait_group<0>();
        fence_proxy_async_smem();                             // images written: visible to the tensor core
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            const uint64_t dM = smem_desc(smem_u32(sm + (mb ? kSoOffM1 : kSoOffM0)), 16384, 1024, kSwizzle128B);
            // D = S^T M^T from (S hi, M hi), (S hi, M lo), (S lo, M hi)
#pragma unroll
            for (int pass = 0; pass < 3; ++pass)
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    umma_f16(tD, dS + (pass == 2 ? uint64_t(kSoImg >> 4) : 0) + uint64_t(((k >> 2) * 16384 + (k & 3) * 32) >> 4),
                             dM + (pass == 1 ? uint64_t(kSoImg >> 4) : 0) + uint64_t((k * 2048) >> 4), id_step,
                             pass > 0 || k > 0);
            umma_commit(&bars[SO_STEP]);
            if (j == nsteps && !to_state) prefetch_tiles(0, 6);
        }
        __syncwarp();
        // while the products run: B_j^T for this thread's TMEM lane and column half
        float b[64];
        so_load_col(slot_of(j), tid & int(kSoEpiThreads - 1), b);   // B_j [dk][dv] (the control warp: unused)
        const bool lf = tid == 0 && !wait(SO_STEP, uint32_t((j - 1) & 1));
        if (__syncthreads_or(lf)) return false;
        if (next_load) load_m(j + 2, mb);
        tc_fence_after();
        float d[64];
        tmem_ld64(tD + lane_addr + uint32_t(half * 64), d);
#pragma unroll
        for (int i = 0; i < 64; ++i) d[i] += b[i];
        if (!epi) {
        } else if (to_state) {                                // S_n: the sequence's final state
            float* dst = p.state_out + (size_t(n) * Hv + h) * kD * kD;
#pragma unroll
            for (int i = 0; i < 64; ++i) dst[size_t(half * 64 + i) * kD + row] = d[i];
        } else {
            so_store_row(sm + kSoOffS, tid, d);
        }
        return true;
    };

    // ---- S_s (or the final state) from S_1 -----------------------------------------
    for (int j = 1; j <= nsteps && !fail; ++j)
        fail = !step(j, (j - 1) & 1, final_role && j == nsteps, j + 2 <= nsteps, j + 1 <= nsteps);
    if (nsteps == 0) cp_async_wait_all();                     // S_1 (and M_1 for a final step)

    // ---- outputs O = O' + G S_s, chunk by chunk ---------------------------------------
    if (!final_role && !fail) {
        if (tid == kSoCtl && !tiles_early) issue_tiles();     // the steps have left the tile region
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == kSoMma) {
            // ---- issuer: products into TMEM buffer i & 1, G tile loads -------------
            {
                const uint32_t id_o = idesc_bf16(128, 64, 0, 0);   // B = G tile, K-major [t][d]
                auto issue_out = [&](int i) {                 // O^T (buffer i & 1) = S^T G^T
                    if (!wait(SO_G0 + i % 3, uint32_t((i / 3) & 1))) return false;
                    // the epilogue has read chunk i - 2 out of this buffer
                    if (i >= 2 && !wait(SO_OFREE0 + (i & 1), uint32_t(((i - 2) >> 1) & 1))) return false;
                    tc_fence_after();
                    const uint64_t dG = smem_desc(smem_u32(sm + kSoOffG + uint32_t(i % 3) * 16384u), 16, 1024, kSwizzle128B);
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        umma_f16(tOb + uint32_t(i & 1) * 64, dS + uint64_t(((k >> 2) * 16384 + (k & 3) * 32) >> 4),
                                 dG + uint64_t(((k >> 2) * 8192 + (k & 3) * 32) >> 4), id_o, k > 0);
                    umma_commit(&bars[SO_O0 + (i & 1)]);
                    return true;
                };
                bool ok = issue_out(0);
                for (int i = 0; i < nout && ok; ++i) {
                    if (i + 1 < nout) ok = issue_out(i + 1);
                    // chunk i's product has read its G tile: the tile takes chunk i + 3
                    if (ok) ok = wait(SO_O0 + (i & 1), uint32_t((i >> 1) & 1));
                    if (ok && i + 3 < nout) issue_g(i + 3);
                }
                if (!ok) *s_err = 1;
            }
        } else if (tid == kSoCtl) {
            // ---- tile thread: stores of the results, O' tile loads ------------------
            {
                bool ok = true;
                for (int i = 0; i < nout; ++i) {
                    if (!wait(SO_STAGED0 + (i & 1), uint32_t((i >> 1) & 1))) {
                        ok = false;
                        break;
                    }
                    if (tile_by_tma(i)) {
                        const uint8_t* ot = sm + kSoOffP + uint32_t(i % 3) * 16384u;
                        const int cs = int(chunk_start(c_lo + i));
                        tma_store_2d(&maps.o, ot, h * kD, cs);
                        tma_store_2d(&maps.o, ot + 8192, h * kD + 64, cs);
                    }
                    bulk_commit_group();
                    // chunk i - 1's store has read its tile: the tile takes chunk i + 2
                    bulk_wait_group_read<1>();
                    if (i + 2 < nout) issue_p(i + 2);
                    prefetch_tiles(i + 6, i + 7);             // and a later chunk's tiles toward L2
                }
                bulk_wait_all();                              // tile stores done before the CTA exits
                if (!ok) *s_err = 1;
            }
        } else if (epi) {
            // ---- epilogue warps: O = O' + (this warp's lanes, token half) ------------
            __nv_bfloat16* gout = static_cast<__nv_bfloat16*>(p.out);
            auto warp_wait = [&](int b, uint32_t parity) {
                bool okw = true;
                if (lane == 0) okw = wait(b, parity);
                return __shfl_sync(0xffffffffu, okw ? 1 : 0, 0) != 0;
            };
            auto warp_arrive = [&](int b) {
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[b]);
            };
            const int m = lane >> 3, rr = lane & 7;
            for (int i = 0; i < nout; ++i) {
                const int bi = i & 1;
                if (!warp_wait(SO_O0 + bi, uint32_t((i >> 1) & 1)) || !warp_wait(SO_P0 + i % 3, uint32_t((i / 3) & 1))) {
                    *s_err = 1;
                    break;
                }
                tc_fence_after();
                uint8_t* ot = sm + kSoOffP + uint32_t(i % 3) * 16384u;   // O' tile, then the result
                // this warp's TMEM lanes (value columns) and token half as 16x256b
                // fragments; O' in the same fragments from its tile; the sum back
                uint32_t r[4][8];
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    tmem_ld_16x256b_x2(tOb + uint32_t(bi * 64) + (uint32_t(quarter * 32 + 16 * (u >> 1)) << 16) +
                                           uint32_t(half * 32 + 16 * (u & 1)),
                                       r[u]);
                tmem_ld_wait();
                tc_fence_before();
                warp_arrive(SO_OFREE0 + bi);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int t = half * 32 + 16 * (u & 1) + 8 * (m >> 1) + rr;
                    const int jj = quarter * 32 + 16 * (u >> 1) + 8 * (m & 1);
                    const uint32_t addr = smem_u32(ot + toff(t, jj, 8192));
                    uint32_t o[4], f[4];
                    ldmatrix_x4_trans(addr, o);
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        f[e] = pack_bf16x2(__uint_as_float(r[u][2 * e]) + __uint_as_float(o[e] << 16),
                                           __uint_as_float(r[u][2 * e + 1]) + __uint_as_float(o[e] & 0xffff0000u));
                    stmatrix_x4_trans(addr, f);
                }
                fence_proxy_async_smem();
                if (!tile_by_tma(i)) {
                    // the chunk ends inside the buffers: this warp's part of the
                    // tile (rows 32 half .., columns 32 quarter ..) as 16-byte rows
                    __syncwarp();
                    const int64_t cs = chunk_start(c_lo + i);
                    const int rows = out_rows(i);
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int idx = lane + 32 * k;
                        const int rw = half * 32 + (idx >> 2), col = quarter * 32 + (idx & 3) * 8;
                        if (rw < rows)
                            *reinterpret_cast<uint4*>(gout + ((cs + rw) * Hv + h) * kD + col) =
                                *reinterpret_cast<const uint4*>(ot + toff(rw, col, 8192));
                    }
                }
                warp_arrive(SO_STAGED0 + bi);
            }
        }
        tc_fence_before();
        __syncthreads();
        if (*s_err) fail = true;
    }
    // the final state here when no CTA of its own forms it: one more step from S_{n-1}
    if (final_after && !fail) {
        if (nsteps > 0) load_m(s, 0);                         // M_1 is still in buffer 0 otherwise
        fail = !step(s, 0, true, false, false);
    }

    // ---- teardown ----------------------------------------------------------------
    cp_async_wait_all();
    tc_fence_before();
    __syncthreads();
    if (tid == kSoMma && (fail || *s_err)) {
        // every output product issued has completed before TMEM goes away
        tc_fence_after();
        umma_commit(&bars[SO_DRAIN]);
        mbar_wait(&bars[SO_DRAIN], 0, kWaitLimit, kSuspendNs);
    }
    if (tid == kSoCtl && (fail || *s_err)) {
        atomicAdd(&g_tc_timeouts, 1);
        // the tile copies still in flight land before shared memory goes away
        const int g_issued = *s_g_issued, p_issued = *s_p_issued;
        for (int i = g_issued - 3 < 0 ? 0 : g_issued - 3; i < g_issued; ++i)
            mbar_wait(&bars[SO_G0 + i % 3], uint32_t((i / 3) & 1), kWaitLimit, kSuspendNs);
        for (int i = p_issued - 3 < 0 ? 0 : p_issued - 3; i < p_issued; ++i)
            mbar_wait(&bars[SO_P0 + i % 3], uint32_t((i / 3) & 1), kWaitLimit, kSuspendNs);
        bulk_wait_all();
    }
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kSoTmemCols);
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

int tc_read_timeouts() {
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_tc_timeouts, sizeof(int)) != cudaSuccess) return -1;
    return v;
}


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
    const bool segmented = p.seg_chunks > 0 && p.seg_max >= 2;
    if ((p.prep_ws != nullptr || segmented) && !make_map(&maps.o, p.out, int64_t(p.Hv) * kD, rows, int64_t(p.Hv) * kD))
        return cudaErrorInvalidValue;
    if (segmented && !make_map(&maps.g, p.g_out, int64_t(p.Hv) * kD, rows, int64_t(p.Hv) * kD))
        return cudaErrorInvalidValue;
    const bool split = p.prep_ws != nullptr && p.prep_slots > 0;
    const void* state_kernel = split ? reinterpret_cast<const void*>(chunk_state_kernel)
                                                     : reinterpret_cast<const void*>(chunk_tc_kernel);
    cudaError_t e = ensure_smem(state_kernel, int(split ? kStSmemBytes : kSmemBytes));
    if (e != cudaSuccess) return e;
    const char* state_name = split ? "chunk_state_kernel" : kTcKernelName;
    auto launch_state = [&](const ChunkParams& q, unsigned z) {
        return split ? launch_pdl(chunk_state_kernel, dim3(q.Hv, q.B, z), kStThreads, kStSmemBytes, s, q, maps)
                     : launch_pdl(chunk_tc_kernel, dim3(q.Hv, q.B, z), kThreads, kSmemBytes, s, q, maps);
    };
    if (split) {                                      // every chunk's S-independent part, in parallel
        if (p.prep_slots > INT32_MAX) return cudaErrorInvalidValue;
        if ((e = ensure_smem(reinterpret_cast<const void*>(chunk_prep_kernel), int(kPrepSmemBytes))) != cudaSuccess)
            return e;
        int dev = 0, sms = 0;
        if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
        if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
        const int64_t items = p.prep_slots * int64_t(p.Hv);
        const int64_t grid = items < 2 * int64_t(sms) ? items : 2 * int64_t(sms);   // two CTAs per SM
        timer_begin(s, "chunk_prep_kernel");
        e = launch_pdl(chunk_prep_kernel, dim3(unsigned(grid)), kPrepThreads, kPrepSmemBytes, s, p, maps);
        timer_end(s);
        if (e != cudaSuccess) return e;
    }
    if (!segmented) {
        ChunkParams q = p;
        q.seg_phase = 0;
        timer_begin(s, state_name);
        e = launch_state(q, 1);
        timer_end(s);
        return e;
    }
    ChunkParams q = p;
    q.seg_phase = 1;                                  // segment 0 in full; O', B_s and G, M_s of the others
    timer_begin(s, state_name);
    e = launch_state(q, unsigned(2 * p.seg_max - 1));
    timer_end(s);
    if (e != cudaSuccess) return e;
    if ((e = ensure_smem(reinterpret_cast<const void*>(seg_out_kernel), int(kSoSmem))) != cudaSuccess) return e;
    timer_begin(s, "seg_out_kernel");                 // S_s, O = O' + G S_s, the final state
    const int so_ctas = p.seg_max - 1 <= kSegTable ? int(p.seg_gstart[p.seg_max - 1]) : (p.seg_max - 1) * p.seg_groups;
    e = launch_pdl(seg_out_kernel, dim3(p.Hv, p.B, unsigned(so_ctas + (p.seg_final_cta ? 1 : 0))), kSoThreads,
                   kSoSmem, s, q, maps);
    timer_end(s);
    return e;
}

}  // namespace gdn
