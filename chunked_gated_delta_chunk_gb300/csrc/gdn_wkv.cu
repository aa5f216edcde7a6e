// RWKV-4 WKV rows ("perf(rwkv): prefill text prompts in multi-token chunks",
// Implementation).  Per channel the state is (num, den, max) with
// A = num exp(max), B = den exp(max) of
//   A_t = exp(w) A_{t-1} + exp(k_t) v_t,   B_t = exp(w) B_{t-1} + exp(k_t),
// and row t outputs wkv_t = (A_{t-1} + exp(u + k_t) v_t) / (B_{t-1} + exp(u + k_t)),
// every exponential taken after subtracting the largest exponent of its sum
// (the decoder's max shift).
//
// The page builds each chunk's rows as a [S + 1, S] exponent tensor; here the
// whole prompt is one HBM-bound pass with the same ticket-ordered tiles and
// decoupled look-back as the selective scan.  Because w does not depend on the
// token, a tile's rows act on an incoming state s as
//   s  ->  decay(s, r w) (+) L,
// with r the tile's row count, decay adding r w to max, (+) the max-shifted sum
// of two states and L the tile's state from an empty start; such maps compose
// in the same form, which is what the look-back combines.  As in the scan, a
// tile has 32 channels (here 128 rows, 32 KB), each warp reduces its 32 rows
// as four interleaved chains, and a sequence start is settled in the first pass: its
// row's output is written there and the state after it replaces the row in
// the staged tile, so no state is read after the first pass.
#include "gdn_common.cuh"
#include "rows_common.cuh"
#include "tc_ptx.cuh"

namespace gdn {

__device__ int g_wkv_timeouts = 0;    // bumped by a CTA whose bounded look-back ran out

namespace {

using namespace ptx;
using rows::find_seq;
using rows::st_release;
constexpr int kCw = rows::kCols;
constexpr float kEmptyMax = -1e38f;

struct St {
    float num, den, mx;
};

// e^x for x <= 0 with the hardware 2^x approximation (relative error about
// 2^-22; results below the smallest normal flush to zero).  Every exponent
// here is a difference from the largest exponent of its sum.
__device__ __forceinline__ float fexp(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x * 1.4426950408889634f));
    return y;
}

__device__ __forceinline__ St empty_state() { return {0.f, 0.f, kEmptyMax}; }

// s after row (k, v): decay by exp(w), then add exp(k) (v, 1)
__device__ __forceinline__ St step(St s, float w, float k, float v) {
    const float ww = s.mx + w;
    const float p = fmaxf(ww, k);
    const float e1 = fexp(ww - p), e2 = fexp(k - p);
    return {fmaf(e1, s.num, e2 * v), fmaf(e1, s.den, e2), p};
}

// (A_{t-1} + exp(u + k) v) / (B_{t-1} + exp(u + k))
__device__ __forceinline__ float output(St s, float u, float k, float v) {
    const float ww = u + k;
    const float p = fmaxf(s.mx, ww);
    const float e1 = fexp(s.mx - p), e2 = fexp(ww - p);
    return __fdividef(fmaf(e1, s.num, e2 * v), fmaf(e1, s.den, e2));
}

// max-shifted sum of two states
__device__ __forceinline__ St add(St a, St b) {
    const float p = fmaxf(a.mx, b.mx);
    const float ea = fexp(a.mx - p), eb = fexp(b.mx - p);
    return {fmaf(ea, a.num, eb * b.num), fmaf(ea, a.den, eb * b.den), p};
}

__device__ __forceinline__ St decay(St s, float x) { return {s.num, s.den, s.mx + x}; }

// The action of some rows on an incoming state s: decay(s, R w) (+) L, or the
// constant L once a sequence starts among the rows (c).
struct Map {
    bool c;
    float R;
    St L;
};

__device__ __forceinline__ Map identity_map() { return {false, 0.f, empty_state()}; }

__device__ __forceinline__ St apply(const Map& m, St s, float w) {
    return m.c ? m.L : add(decay(s, m.R * w), m.L);
}

// m2 after m1
__device__ __forceinline__ Map compose(const Map& m2, const Map& m1, float w) {
    if (m2.c) return m2;
    return {m1.c, m1.R + m2.R, add(decay(m1.L, m2.R * w), m2.L)};
}

__device__ __forceinline__ St load_state(const float* base, int64_t n, int C, int c) {
    if (base == nullptr) return empty_state();
    return {base[(n * 3 + 0) * C + c], base[(n * 3 + 1) * C + c], base[(n * 3 + 2) * C + c]};
}

__device__ __forceinline__ void store_state(float* base, int64_t n, int C, int c, St s) {
    base[(n * 3 + 0) * C + c] = s.num;
    base[(n * 3 + 1) * C + c] = s.den;
    base[(n * 3 + 2) * C + c] = s.mx;
}

// Workspace vectors of a tile: (num, den, max) of its map's L, then of its end state.
__device__ __forceinline__ void put(float* v, size_t tiles, size_t slot, St s) {
    v[slot] = s.num;
    v[tiles * kCw + slot] = s.den;
    v[2 * tiles * kCw + slot] = s.mx;
}
__device__ __forceinline__ St get(const float* v, size_t tiles, size_t slot) {
    return {__ldcg(v + slot), __ldcg(v + tiles * kCw + slot), __ldcg(v + 2 * tiles * kCw + slot)};
}

__global__ void wkv_init_kernel(const WkvParams p) {
    griddep_wait();                                   // the grid before may still use the flags
    const int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i == 0) *p.ticket = 0;
    if (i < p.n_tiles) p.flags[i] = 0;
    if (i < int64_t(p.B) * p.C) {
        const int n = int(i / p.C), c = int(i % p.C);
        if (p.cu[n + 1] <= p.cu[n]) store_state(p.state_out, n, p.C, c, load_state(p.state_in, n, p.C, c));
    }
}

__global__ void __launch_bounds__(rows::kThreads) wkv_rows_kernel(const WkvParams p) {
    griddep_wait();                                   // ticket and flags from wkv_init_kernel
    using namespace rows;
    constexpr int kRows = rows::kWkvRows;             // rows of a tile
    constexpr int kWarpRows = kRows / kWarps;         // rows of a warp
    constexpr int kChainRows = kWarpRows / kChains;   // rows of one of a thread's chains
    extern __shared__ __align__(16) float sm_wkv[];
    float* sk = sm_wkv;                               // [kRows][kCols]
    float* sv = sm_wkv + kRows * kCols;
    __shared__ int s_tile;
    __shared__ int s_seq[kRows], s_mark[kRows];
    __shared__ float s_R[kWarps][kCols], s_L[3][kWarps][kCols], s_in[3][kWarps][kCols];
    __shared__ int s_first[kWarps];                   // first start row of each warp, or -1
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) s_tile = atomicAdd(p.ticket, 1);
    __syncthreads();
    const int tile = s_tile;
    const int ci = tile / p.n_cb, cb = tile % p.n_cb;
    const int64_t t0 = int64_t(ci) * kRows;
    const int nrow = int(p.T - t0 < kRows ? p.T - t0 : kRows);
    const int c0 = cb * kCols, c = c0 + lane;
    const bool live = c < p.C;
    const size_t tiles = size_t(p.n_tiles);
    stage_tile<kRows>(sk, sv, p.k, p.v, t0, nrow, c0, p.C, tid);
    const float w = live ? p.w[c] : 0.f, u = live ? p.u[c] : 0.f;
    fill_row_info(p.cu, p.B, t0, nrow, tid, s_seq, s_mark);
    cp_async_wait_all();
    __syncthreads();

    // ---- pass 1: the map of each chain of the warp's rows.  A start row's
    // output is written here, and the state after it replaces (k, v) in the
    // staged tile as (max + log den, num / den), the same state with den = 1.
    Map M[kChains];
#pragma unroll
    for (int j = 0; j < kChains; ++j) M[j] = identity_map();
    int first = -1;
    const int rw = warp * kWarpRows;
#pragma unroll 4
    for (int i = 0; i < kChainRows; ++i) {
#pragma unroll
        for (int j = 0; j < kChains; ++j) {
            const int r = rw + j * kChainRows + i;
            if (r < nrow) {
                const float kt = sk[r * kCols + lane], vt = sv[r * kCols + lane];
                if (s_mark[r] & kRowStart) {
                    const int n = s_seq[r];
                    const St s0 = live ? load_state(p.state_in, n, p.C, c) : empty_state();
                    const St s1 = step(s0, w, kt, vt);
                    if (live) p.wkv[(t0 + r) * p.C + c] = output(s0, u, kt, vt);
                    sk[r * kCols + lane] = s1.mx + logf(s1.den);
                    sv[r * kCols + lane] = s1.num / s1.den;
                    M[j] = {true, 0.f, s1};
                    if (first < 0 || r < first) first = r;
                } else {
                    M[j].L = step(M[j].L, w, kt, vt);
                    M[j].R += 1.f;
                }
            }
        }
    }
    {
        Map Mw = M[0];
#pragma unroll
        for (int j = 1; j < kChains; ++j) Mw = compose(M[j], Mw, w);
        s_R[warp][lane] = Mw.c ? -1.f : Mw.R;         // -1 marks a constant map
        s_L[0][warp][lane] = Mw.L.num;
        s_L[1][warp][lane] = Mw.L.den;
        s_L[2][warp][lane] = Mw.L.mx;
        if (lane == 0) s_first[warp] = first;
    }
    __syncthreads();

    // ---- warp 0: publish, look back, hand out the warps' incoming states ------
    if (warp == 0) {
        auto warp_map = [&](int v) {
            const float R = s_R[v][lane];
            return Map{R < 0.f, R < 0.f ? 0.f : R, St{s_L[0][v][lane], s_L[1][v][lane], s_L[2][v][lane]}};
        };
        Map Mt = warp_map(0);
#pragma unroll
        for (int v = 1; v < kWarps; ++v) Mt = compose(warp_map(v), Mt, w);
        const bool reset = Mt.c;
        const size_t slot = size_t(tile) * kCols + lane;
        if (reset) put(p.incl, tiles, slot, Mt.L);    // end state known: no carry reaches it
        else put(p.agg, tiles, slot, Mt.L);
        __threadfence();
        __syncwarp();
        if (lane == 0) st_release(&p.flags[tile], reset ? 2 : 1);
        St x = empty_state();
        bool fail = false;
        if (s_first[0] != 0) {                        // row 0 continues the previous tile
            float R = 0.f;                            // carry map: y -> decay(y, R w) (+) L
            St L = empty_state();
            bool done = false;
            for (int pci = ci - 1; pci >= 0 && !done; --pci) {
                const int pidx = pci * p.n_cb + cb;
                int f = 0;
                if (lane == 0) f = wait_flag(&p.flags[pidx]);
                __syncwarp();
                f = __shfl_sync(0xffffffffu, f, 0);
                if (f == 0) {
                    fail = true;
                    break;
                }
                const size_t ps = size_t(pidx) * kCols + lane;
                if (f == 2) {
                    x = add(decay(get(p.incl, tiles, ps), R * w), L);
                    done = true;
                } else {
                    const int prow = int(p.T - int64_t(pci) * kRows < kRows ? p.T - int64_t(pci) * kRows : kRows);
                    L = add(decay(get(p.agg, tiles, ps), R * w), L);
                    R += float(prow);
                }
            }
            if (!done && !fail) x = L;                // no predecessor (malformed cu_seqlens)
        }
        if (!reset) {
            put(p.incl, tiles, slot, apply(Mt, x, w));
            __threadfence();
            __syncwarp();
            if (lane == 0) st_release(&p.flags[tile], 2);
        }
        if (fail && lane == 0) atomicAdd(&g_wkv_timeouts, 1);
#pragma unroll
        for (int v = 0; v < kWarps; ++v) {
            s_in[0][v][lane] = x.num;
            s_in[1][v][lane] = x.den;
            s_in[2][v][lane] = x.mx;
            x = apply(warp_map(v), x, w);
        }
    }
    __syncthreads();

    // ---- pass 2: outputs from the staged rows, each chain from its own input --
    if (!live) return;
    St st[kChains];
    st[0] = St{s_in[0][warp][lane], s_in[1][warp][lane], s_in[2][warp][lane]};
#pragma unroll
    for (int j = 1; j < kChains; ++j) st[j] = apply(M[j - 1], st[j - 1], w);
#pragma unroll 4
    for (int i = 0; i < kChainRows; ++i) {
#pragma unroll
        for (int j = 0; j < kChains; ++j) {
            const int r = rw + j * kChainRows + i;
            if (r < nrow) {
                const int mark = s_mark[r];
                const float kt = sk[r * kCols + lane], vt = sv[r * kCols + lane];
                if (mark & kRowStart) {
                    st[j] = St{vt, 1.f, kt};          // the state after the start row (pass 1)
                } else {
                    p.wkv[(t0 + r) * p.C + c] = output(st[j], u, kt, vt);
                    st[j] = step(st[j], w, kt, vt);
                }
                if (mark & kRowEnd) store_state(p.state_out, s_seq[r], p.C, c, st[j]);
            }
        }
    }
}

}  // namespace

size_t wkv_workspace_bytes(int C, int64_t T) {
    const int64_t tiles = ((T + rows::kWkvRows - 1) / rows::kWkvRows) * ((C + kCw - 1) / kCw);
    auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
    return up(sizeof(int)) + up(size_t(tiles) * sizeof(int)) + 2 * up(size_t(tiles) * kCw * 3 * sizeof(float));
}

void wkv_bind_workspace(WkvParams& p, void* ws) {
    auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
    char* w = static_cast<char*>(ws);
    p.n_cb = (p.C + kCw - 1) / kCw;
    p.n_tiles = int(((p.T + rows::kWkvRows - 1) / rows::kWkvRows) * p.n_cb);
    p.ticket = reinterpret_cast<int*>(w);
    w += up(sizeof(int));
    p.flags = reinterpret_cast<int*>(w);
    w += up(size_t(p.n_tiles) * sizeof(int));
    const size_t vec = up(size_t(p.n_tiles) * kCw * 3 * sizeof(float));
    p.agg = reinterpret_cast<float*>(w);
    p.incl = reinterpret_cast<float*>(w + vec);
}

cudaError_t launch_wkv_rows(const WkvParams& p, cudaStream_t s) {
    const int64_t init_items = int64_t(p.B) * p.C > p.n_tiles ? int64_t(p.B) * p.C : p.n_tiles;
    if (init_items > 0) {
        timer_begin(s, "wkv_init_kernel");
        cudaError_t e = launch_pdl(wkv_init_kernel, dim3(unsigned((init_items + 255) / 256)), 256, 0, s, p);
        timer_end(s);
        if (e != cudaSuccess) return e;
    }
    if (p.n_tiles == 0) return cudaSuccess;
    const int smem = 2 * rows::kWkvRows * kCw * int(sizeof(float));
    cudaError_t e = ensure_smem(reinterpret_cast<const void*>(wkv_rows_kernel), smem);
    if (e != cudaSuccess) return e;
    timer_begin(s, "wkv_rows_kernel");
    e = launch_pdl(wkv_rows_kernel, dim3(unsigned(p.n_tiles)), rows::kThreads, unsigned(smem), s, p);
    timer_end(s);
    return e;
}

int wkv_read_timeouts() {
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_wkv_timeouts, sizeof(int)) != cudaSuccess) return -1;
    return v;
}

}  // namespace gdn
