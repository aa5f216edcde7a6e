// Full-attention rows over a KV cache plus the chunk's causal prefix
// ("perf(qwen3_5): prefill text prompts in multi-token chunks",
// Implementation: the full-attention layers of a prefill chunk attend over
// the cache plus the chunk's causal prefix, and the chunk's present k / v
// rows are appended to the cache).
//
// attn_append_kernel writes the prompt's k, v rows into the cache after each
// sequence's cache_len rows.  attn_rows_kernel then runs one CTA per
// (128-row query tile, query head, sequence), warp-specialised:
//   warp 8      TMA: the query tile once, key tiles (2 stages) and value
//               tiles (3 stages) of 128 rows from the cache;
//   warp 9      tcgen05 MMAs: S_j = Q K_j^T into one of two TMEM buffers, then
//               O += P_{j-1} V_{j-1} with P (bf16, two TMEM buffers) as the A
//               operand from TMEM;
//   warps 0-7   softmax, two threads per query row (its TMEM lane), one per
//               half of the keys: causal / capacity mask, running maximum
//               (raised, with O and l rescaled, only past 2^8 of headroom),
//               P = exp2(S scale - m) into TMEM.
// mbarriers hand every buffer between the roles, so the MMAs of tile j + 1
// run while tile j's softmax is computed.
#include <cuda.h>
#include <climits>

#include "gdn_common.cuh"
#include "tc_ptx.cuh"

namespace gdn {

__device__ int g_attn_timeouts = 0;   // bumped by a CTA whose bounded wait ran out

namespace {

using namespace ptx;

constexpr int kAD = 128;              // head dim
constexpr int kAQ = 128;              // query rows per tile (TMEM lanes)
constexpr int kAK = 128;              // keys per tile
// K_j is needed by S_j early in a tile and V_j by O += P_j V_j at its end, so
// values get the deeper buffering: a key tile refills after S_{j-2}, a value
// tile after the product of tile j - 3.
constexpr int kAKStages = 2, kAVStages = 3;
constexpr int kASoftThreads = 256;    // warps 0-7
constexpr int kAThreads = kASoftThreads + 64;   // + TMA warp + MMA warp
constexpr uint32_t kAWaitLimit = 1u << 20;
// The pipeline's hand-offs are short: waits re-check every ~32 ns instead of
// sleeping up to the default 2 us (the bound stays well under a second).
constexpr uint32_t kASuspendNs = 32, kASpinLimit = 1u << 24;
constexpr float kARescale = 8.f;      // log2 headroom before the reference maximum moves
constexpr uint32_t kATile = kAK * kAD * 2;                 // 32 KB per Q, K or V tile
constexpr uint32_t kAOffQ = 0;
constexpr uint32_t kAOffK = kATile;
constexpr uint32_t kAOffV = kAOffK + kAKStages * kATile;
constexpr uint32_t kAOffBar = kAOffV + kAVStages * kATile;
constexpr uint32_t kANumBars = 19;
constexpr uint32_t kAOffEx = kAOffBar + 256;               // [2 parities][2 halves][kAQ] floats: maxima
constexpr uint32_t kAOffL = kAOffEx + 2 * 2 * kAQ * 4;     // [2 halves][kAQ] floats: row sums
constexpr uint32_t kASmem = kAOffL + 2 * kAQ * 4 + 1024;
static_assert(kASmem <= 232448, "attention stages above the 227 KB per-block limit");
// TMEM: S in two buffers (2 x 128 columns), P (bf16 pairs) in two buffers
// (2 x 64), O (128)
constexpr uint32_t kAColS = 0, kAColP = 256, kAColO = 384, kATmemCols = 512;
enum : int {
    AB_Q = 0,
    AB_KFULL = 1,                     // + key stage
    AB_KEMPTY = AB_KFULL + kAKStages,
    AB_VFULL = AB_KEMPTY + kAKStages, // + value stage
    AB_VEMPTY = AB_VFULL + kAVStages,
    AB_SFULL = AB_VEMPTY + kAVStages, // + S buffer (2)
    AB_SEMPTY = AB_SFULL + 2,         // + S buffer (2), 8 arrivals
    AB_PFULL = AB_SEMPTY + 2,         // + P buffer (2), 8 arrivals
    AB_ODONE = AB_PFULL + 2           // + P buffer (2): O += P V of that buffer done
};
static_assert(AB_ODONE + 2 == int(kANumBars), "barrier count");

struct AttnMaps {
    CUtensorMap q, kc, vc;
};

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ int attn_find_seq(const int32_t* cu, int B, int64_t t) {
    int lo = 0, hi = B - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (int64_t(cu[mid]) <= t) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

// Prompt rows into the cache: row t of sequence n goes to position
// cache_len[n] + (t - cu[n]) (rows past the capacity are dropped).
__global__ void attn_append_kernel(const AttnParams p) {
    griddep_wait();                                   // the grid before may still read the cache
    const int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;   // (t, kv head, 16-byte word)
    const int words = kAD / 8;
    if (i >= p.T * p.Hkv * words) return;
    const int64_t t = i / (int64_t(p.Hkv) * words);
    const int kh = int(i / words % p.Hkv), w = int(i % words);
    const int n = attn_find_seq(p.cu, p.B, t);
    const int64_t pos = int64_t(p.cache_len[n]) + (t - p.cu[n]);
    if (pos < 0 || pos >= p.cap) return;
    const size_t src = (size_t(t) * p.Hkv + kh) * kAD + w * 8;
    const size_t dst = ((size_t(n) * p.Hkv + kh) * p.cap + pos) * kAD + w * 8;
    const __nv_bfloat16* k = static_cast<const __nv_bfloat16*>(p.k);
    const __nv_bfloat16* v = static_cast<const __nv_bfloat16*>(p.v);
    *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.k_cache) + dst) = *reinterpret_cast<const uint4*>(k + src);
    *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.v_cache) + dst) = *reinterpret_cast<const uint4*>(v + src);
}

__global__ void __launch_bounds__(kAThreads, 1)
attn_rows_kernel(const AttnParams p, const __grid_constant__ AttnMaps maps) {
    griddep_wait();                                   // the cache rows attn_append_kernel wrote
    extern __shared__ uint8_t attn_smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(attn_smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kAOffBar);
    float* s_ex = reinterpret_cast<float*>(sm + kAOffEx);
    float* s_l = reinterpret_cast<float*>(sm + kAOffL);
    __shared__ uint32_t tmem_slot;
    __shared__ volatile int s_fail;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h = blockIdx.y, n = blockIdx.z;
    const int xt = int(gridDim.x) - 1 - int(blockIdx.x);          // long (late) tiles first
    const int64_t s0 = p.cu[n];
    const int L = int(p.cu[n + 1] - s0);
    const int q0 = xt * kAQ;
    if (q0 >= L) return;                                          // the whole CTA leaves together
    const int rows = L - q0 < kAQ ? L - q0 : kAQ;
    const int clen = p.cache_len[n];
    const int kh = h / (p.Hq / p.Hkv);
    int nkeys = clen + q0 + rows;                                 // keys the tile's last row sees
    if (nkeys > p.cap) nkeys = p.cap;
    const int ntiles = (nkeys + kAK - 1) / kAK;
    const int kv_row0 = int((int64_t(n) * p.Hkv + kh) * p.cap);

    if (tid == 0) {
        for (int i = 0; i < int(kANumBars); ++i)
            mbar_init(&bars[i], (i == AB_SEMPTY || i == AB_SEMPTY + 1 || i == AB_PFULL || i == AB_PFULL + 1) ? 8 : 1);
        fence_mbar_init();
        s_fail = 0;
    }
    if (warp == 0) {
        tmem_alloc(&tmem_slot, kATmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    const uint32_t tP = tmem + kAColP, tO = tmem + kAColO;
    auto wait = [&](int b, uint32_t parity) {
        if (s_fail) return false;
        if (mbar_wait(&bars[b], parity, kASpinLimit, kASuspendNs)) return true;
        s_fail = 1;
        return false;
    };

    if (warp == 8) {
        // ================================================================ TMA
        if (lane == 0) {
            tma_prefetch_desc(&maps.q);
            tma_prefetch_desc(&maps.kc);
            tma_prefetch_desc(&maps.vc);
            uint8_t* sQ = sm + kAOffQ;
            mbar_arrive_expect_tx(&bars[AB_Q], kATile);
            tma_load_2d(sQ, &maps.q, &bars[AB_Q], h * kAD, int(s0 + q0));
            tma_load_2d(sQ + kATile / 2, &maps.q, &bars[AB_Q], h * kAD + 64, int(s0 + q0));
            int k_last[kAKStages], v_last[kAVStages];
            for (int st = 0; st < kAKStages; ++st) k_last[st] = -1;
            for (int st = 0; st < kAVStages; ++st) v_last[st] = -1;
            for (int j = 0; j < ntiles; ++j) {
                const int ks = j % kAKStages, vs = j % kAVStages, y = kv_row0 + j * kAK;
                if (j >= kAKStages && !wait(AB_KEMPTY + ks, uint32_t((j / kAKStages - 1) & 1))) break;
                uint8_t* dk = sm + kAOffK + ks * kATile;
                mbar_arrive_expect_tx(&bars[AB_KFULL + ks], kATile);
                tma_load_2d(dk, &maps.kc, &bars[AB_KFULL + ks], 0, y);
                tma_load_2d(dk + kATile / 2, &maps.kc, &bars[AB_KFULL + ks], 64, y);
                k_last[ks] = j;
                if (j >= kAVStages && !wait(AB_VEMPTY + vs, uint32_t((j / kAVStages - 1) & 1))) break;
                uint8_t* dv = sm + kAOffV + vs * kATile;
                mbar_arrive_expect_tx(&bars[AB_VFULL + vs], kATile);
                tma_load_2d(dv, &maps.vc, &bars[AB_VFULL + vs], 0, y);
                tma_load_2d(dv + kATile / 2, &maps.vc, &bars[AB_VFULL + vs], 64, y);
                v_last[vs] = j;
            }
            if (s_fail) {
                // let the copies still in flight land before shared memory goes away
                mbar_wait(&bars[AB_Q], 0, kAWaitLimit);
                for (int st = 0; st < kAKStages; ++st)
                    if (k_last[st] >= 0) mbar_wait(&bars[AB_KFULL + st], uint32_t((k_last[st] / kAKStages) & 1), kAWaitLimit);
                for (int st = 0; st < kAVStages; ++st)
                    if (v_last[st] >= 0) mbar_wait(&bars[AB_VFULL + st], uint32_t((v_last[st] / kAVStages) & 1), kAWaitLimit);
            }
        }
        __syncwarp();
    } else if (warp == 9) {
        // ================================================================ MMA
        if (lane == 0) {
            const uint32_t id_s = idesc_bf16(kAQ, kAK, 0, 0);     // B = K, K-major
            const uint32_t id_o = idesc_bf16(kAQ, kAD, 0, 1);     // B = V, MN-major [key][d]
            const uint64_t dq = smem_desc(smem_u32(sm + kAOffQ), 16, 1024, kSwizzle128B);
            auto issue_pv = [&](int j) {                          // O += P_j V_j
                if (!wait(AB_VFULL + j % kAVStages, uint32_t((j / kAVStages) & 1))) return false;
                if (!wait(AB_PFULL + (j & 1), uint32_t((j >> 1) & 1))) return false;
                tc_fence_after();
                const uint64_t dv = smem_desc(smem_u32(sm + kAOffV + (j % kAVStages) * kATile), kATile / 2, 1024,
                                              kSwizzle128B);
#pragma unroll
                for (int s = 0; s < kAK / 16; ++s)
                    umma_f16_tmemA(tO, tP + uint32_t(j & 1) * (kAK / 2) + s * 8, dv + uint64_t(s * 2048 >> 4), id_o,
                                   j > 0 || s > 0);
                umma_commit(&bars[AB_ODONE + (j & 1)]);
                umma_commit(&bars[AB_VEMPTY + j % kAVStages]);
                return true;
            };
            bool ok = wait(AB_Q, 0);
            for (int j = 0; ok && j < ntiles; ++j) {
                const int b = j & 1;
                ok = wait(AB_KFULL + j % kAKStages, uint32_t((j / kAKStages) & 1));
                if (ok && j >= 2) ok = wait(AB_SEMPTY + b, uint32_t(((j >> 1) - 1) & 1));
                if (!ok) break;
                tc_fence_after();
                const uint64_t dk = smem_desc(smem_u32(sm + kAOffK + (j % kAKStages) * kATile), 16, 1024, kSwizzle128B);
#pragma unroll
                for (int s = 0; s < kAD / 16; ++s) {
                    const uint32_t off = uint32_t(s >> 2) * (kATile / 2) + uint32_t(s & 3) * 32u;
                    umma_f16(tmem + kAColS + b * kAK, dq + (off >> 4), dk + (off >> 4), id_s, s > 0);
                }
                umma_commit(&bars[AB_SFULL + b]);
                umma_commit(&bars[AB_KEMPTY + j % kAKStages]);
                if (j >= 1) ok = issue_pv(j - 1);
            }
            if (ok && ntiles > 0) issue_pv(ntiles - 1);
        }
        __syncwarp();
    } else {
        // ================================================================ softmax
        const int row = (warp & 3) * 32 + lane;                   // TMEM lane = query row
        const int half = warp >> 2;                               // keys 64 half .. 64 half + 63
        const uint32_t lane_addr = uint32_t((warp & 3) * 32) << 16;
        const uint32_t pair_bar = 1 + (warp & 3);                 // warps w and w + 4 share the rows
        const float sl2 = p.scale * 1.4426950408889634f;
        const int pos = clen + q0 + row;                          // this row sees keys 0 .. pos
        float m_ref = -INFINITY, l = 0.f;
        bool fail = false;
        for (int j = 0; j < ntiles; ++j) {
            const int b = j & 1;
            if (lane == 0) fail = fail || !wait(AB_SFULL + b, uint32_t((j >> 1) & 1));
            __syncwarp();
            fail = __shfl_sync(0xffffffffu, fail, 0);
            tc_fence_after();
            float x[kAK / 2];
            if (!fail) {
#pragma unroll
                for (int q = 0; q < kAK / 2; q += 32) {
                    uint32_t r0[16], r1[16];
                    const uint32_t ta = tmem + kAColS + b * kAK + lane_addr + half * (kAK / 2) + q;
                    GDN_TMEM_LD_X16(ta, r0);
                    GDN_TMEM_LD_X16(ta + 16, r1);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        x[q + i] = __uint_as_float(r0[i]);
                        x[q + 16 + i] = __uint_as_float(r1[i]);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[AB_SEMPTY + b]);     // this warp is done with S_j
            // ---- mask and the half-row maximum (raw scores; the scale is
            // positive, so it is applied to the maximum); the pair agrees on the
            // row's maximum.  Key tiles that every row of this warp sees whole
            // skip the mask.
            const int k0 = j * kAK + half * (kAK / 2);
            const bool whole = k0 + kAK / 2 - 1 <= clen + q0 + (warp & 3) * 32 && k0 + kAK / 2 <= nkeys;
            if (fail || !whole) {
#pragma unroll
                for (int c = 0; c < kAK / 2; ++c) {
                    const int kk = k0 + c;
                    x[c] = (!fail && kk <= pos && kk < nkeys) ? x[c] : -INFINITY;
                }
            }
            float mq[4] = {x[0], x[1], x[2], x[3]};
#pragma unroll
            for (int c = 4; c < kAK / 2; ++c) mq[c & 3] = fmaxf(mq[c & 3], x[c]);
            const float mh = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3])) * sl2;
            s_ex[(b * 2 + half) * kAQ + row] = mh;
            if (named_sync_or(pair_bar, 64, fail)) {
                fail = true;
                break;
            }
            const float mt = fmaxf(s_ex[(b * 2) * kAQ + row], s_ex[(b * 2 + 1) * kAQ + row]);
            float f = 1.f;                                        // rescale of O and l
            if (j == 0) {
                m_ref = mt;
            } else if (mt > m_ref + kARescale) {
                f = ex2(m_ref - mt);
                m_ref = mt;
            }
            // P = exp2(scale x - m_ref) as one multiply-add and one 2^x each;
            // the row sum gathers the fp32 values
            uint32_t pk[kAK / 4];
            float lq[4] = {0.f, 0.f, 0.f, 0.f};
            const float nm = -m_ref;
#pragma unroll
            for (int c = 0; c < kAK / 2; c += 2) {
                const float e0 = ex2(fmaf(x[c], sl2, nm)), e1 = ex2(fmaf(x[c + 1], sl2, nm));
                pk[c / 2] = pack2(e0, e1);
                lq[(c >> 1) & 3] += e0 + e1;
            }
            l = fmaf(l, f, (lq[0] + lq[1]) + (lq[2] + lq[3]));
            // ---- P_j goes to buffer j & 1 once O += P_{j-2} V_{j-2} is done; O is
            // rescaled (rarely) once every product so far is in ---------------
            const bool resc = __any_sync(0xffffffffu, f != 1.f);
            if (lane == 0 && j >= 2) fail = fail || !wait(AB_ODONE + b, uint32_t(((j - 2) >> 1) & 1));
            if (lane == 0 && resc && j >= 1) fail = fail || !wait(AB_ODONE + ((j - 1) & 1), uint32_t(((j - 1) >> 1) & 1));
            __syncwarp();
            fail = __shfl_sync(0xffffffffu, fail, 0);
            tc_fence_after();
            if (!fail && resc) {                                  // rescale this warp's half rows of O
#pragma unroll
                for (int q = 0; q < kAD / 2; q += 16) {
                    float o[16];
                    tmem_ld16(tO + lane_addr + half * (kAD / 2) + q, o);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 16; ++i) o[i] *= f;
                    tmem_st16(tO + lane_addr + half * (kAD / 2) + q, o);
                }
            }
            if (!fail) {
#pragma unroll
                for (int q = 0; q < kAK / 4; q += 16) {
                    __syncwarp();
                    GDN_TMEM_ST_X16(tP + uint32_t(b) * (kAK / 2) + lane_addr + half * (kAK / 4) + q, (pk + q));
                }
                tmem_st_wait();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[AB_PFULL + b]);
        }
        // ---- O / l to the output rows -------------------------------------------
        if (lane == 0 && !fail && ntiles > 0)
            fail = !wait(AB_ODONE + ((ntiles - 1) & 1), uint32_t(((ntiles - 1) >> 1) & 1));
        __syncwarp();
        fail = __shfl_sync(0xffffffffu, fail, 0);
        s_l[half * kAQ + row] = l;
        if (!named_sync_or(pair_bar, 64, fail)) {
            tc_fence_after();
            const float inv = 1.f / (s_l[row] + s_l[kAQ + row]);
            __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.o) + ((s0 + q0 + row) * p.Hq + h) * kAD + half * (kAD / 2);
#pragma unroll
            for (int q = 0; q < kAD / 2; q += 16) {
                float o[16];
                tmem_ld16(tO + lane_addr + half * (kAD / 2) + q, o);
                tmem_ld_wait();
                uint4 w0, w1;
                w0.x = pack2(o[0] * inv, o[1] * inv);
                w0.y = pack2(o[2] * inv, o[3] * inv);
                w0.z = pack2(o[4] * inv, o[5] * inv);
                w0.w = pack2(o[6] * inv, o[7] * inv);
                w1.x = pack2(o[8] * inv, o[9] * inv);
                w1.y = pack2(o[10] * inv, o[11] * inv);
                w1.z = pack2(o[12] * inv, o[13] * inv);
                w1.w = pack2(o[14] * inv, o[15] * inv);
                if (row < rows) {
                    *reinterpret_cast<uint4*>(out + q) = w0;
                    *reinterpret_cast<uint4*>(out + q + 8) = w1;
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (tid == 0 && s_fail) atomicAdd(&g_attn_timeouts, 1);
    if (warp == 0) tmem_dealloc(tmem, kATmemCols);
}

typedef CUresult (*AttnEncodeFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                 CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                 CUtensorMapFloatOOBfill);

AttnEncodeFn attn_encode_fn() {
    static AttnEncodeFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        cudaDriverEntryPointQueryResult q;
        void* f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<AttnEncodeFn>(f);
    }
    return fn;
}

// bf16 rows of `width` elements, row pitch `pitch` elements; boxes of
// 64 columns x 128 rows with the 128-byte swizzle.
bool attn_map(CUtensorMap* m, const void* base, int64_t width, int64_t rows, int64_t pitch) {
    AttnEncodeFn enc = attn_encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {cuuint64_t(width), cuuint64_t(rows)};
    cuuint64_t strides[1] = {cuuint64_t(pitch) * 2};
    cuuint32_t box[2] = {64, 128};
    cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_attn_rows(const AttnParams& p, cudaStream_t s) {
    if (p.B == 0) return cudaSuccess;
    if (p.T > 0) {
        const int64_t items = p.T * p.Hkv * (kAD / 8);
        timer_begin(s, "attn_append_kernel");
        cudaError_t e = launch_pdl(attn_append_kernel, dim3(unsigned((items + 255) / 256)), 256, 0, s, p);
        timer_end(s);
        if (e != cudaSuccess) return e;
    }
    if (p.T == 0) return cudaSuccess;
    AttnMaps maps;
    const int64_t cache_rows = int64_t(p.B) * p.Hkv * p.cap;
    if (cache_rows > INT32_MAX || p.T > INT32_MAX) return cudaErrorInvalidValue;
    if (!attn_map(&maps.q, p.q, int64_t(p.Hq) * kAD, p.T, int64_t(p.Hq) * kAD) ||
        !attn_map(&maps.kc, p.k_cache, kAD, cache_rows, kAD) || !attn_map(&maps.vc, p.v_cache, kAD, cache_rows, kAD))
        return cudaErrorInvalidValue;
    cudaError_t e = ensure_smem(reinterpret_cast<const void*>(attn_rows_kernel), int(kASmem));
    if (e != cudaSuccess) return e;
    const unsigned qtiles = unsigned((p.max_len + kAQ - 1) / kAQ);
    if (qtiles == 0) return cudaSuccess;
    timer_begin(s, "attn_rows_kernel");
    e = launch_pdl(attn_rows_kernel, dim3(qtiles, p.Hq, p.B), kAThreads, kASmem, s, p, maps);
    timer_end(s);
    return e;
}

int attn_read_timeouts() {
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_attn_timeouts, sizeof(int)) != cudaSuccess) return -1;
    return v;
}

}  // namespace gdn
