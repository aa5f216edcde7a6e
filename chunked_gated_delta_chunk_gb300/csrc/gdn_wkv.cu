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
// in the same form, which is what the look-back combines.
#include "gdn_common.cuh"
#include "rows_common.cuh"
#include "tc_ptx.cuh"

namespace gdn {

__device__ int g_wkv_timeouts = 0;    // bumped by a CTA whose bounded look-back ran out

namespace {

using namespace ptx;
using rows::find_seq;
using rows::st_release;
constexpr int kR = rows::kRows, kCw = rows::kCols;
constexpr float kEmptyMax = -1e38f;

struct St {
    float num, den, mx;
};

__device__ __forceinline__ St empty_state() { return {0.f, 0.f, kEmptyMax}; }

// s after row (k, v): decay by exp(w), then add exp(k) (v, 1)
__device__ __forceinline__ St step(St s, float w, float k, float v) {
    const float ww = s.mx + w;
    const float p = fmaxf(ww, k);
    const float e1 = expf(ww - p), e2 = expf(k - p);
    return {fmaf(e1, s.num, e2 * v), fmaf(e1, s.den, e2), p};
}

// (A_{t-1} + exp(u + k) v) / (B_{t-1} + exp(u + k))
__device__ __forceinline__ float output(St s, float u, float k, float v) {
    const float ww = u + k;
    const float p = fmaxf(s.mx, ww);
    const float e1 = expf(s.mx - p), e2 = expf(ww - p);
    return fmaf(e1, s.num, e2 * v) / fmaf(e1, s.den, e2);
}

// max-shifted sum of two states
__device__ __forceinline__ St add(St a, St b) {
    const float p = fmaxf(a.mx, b.mx);
    const float ea = expf(a.mx - p), eb = expf(b.mx - p);
    return {fmaf(ea, a.num, eb * b.num), fmaf(ea, a.den, eb * b.den), p};
}

__device__ __forceinline__ St decay(St s, float x) { return {s.num, s.den, s.mx + x}; }

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
    const int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i == 0) *p.ticket = 0;
    if (i < p.n_tiles) p.flags[i] = 0;
    if (i < int64_t(p.B) * p.C) {
        const int n = int(i / p.C), c = int(i % p.C);
        if (p.cu[n + 1] <= p.cu[n]) store_state(p.state_out, n, p.C, c, load_state(p.state_in, n, p.C, c));
    }
}

__global__ void __launch_bounds__(kCw) wkv_rows_kernel(const WkvParams p) {
    extern __shared__ __align__(16) float sm_wkv[];
    float* sk = sm_wkv;                               // [kR][kCw]
    float* sv = sm_wkv + kR * kCw;
    __shared__ int s_tile, s_flag, s_fail;
    const int tid = threadIdx.x;
    if (tid == 0) {
        s_tile = atomicAdd(p.ticket, 1);
        s_fail = 0;
    }
    __syncthreads();
    const int tile = s_tile;
    const int ci = tile / p.n_cb, cb = tile % p.n_cb;
    const int64_t t0 = int64_t(ci) * kR;
    const int nrow = int(p.T - t0 < kR ? p.T - t0 : kR);
    const int c0 = cb * kCw, c = c0 + tid;
    const bool live = c < p.C;
    const size_t tiles = size_t(p.n_tiles);

    for (int i = tid; i < kR * (kCw / 4); i += kCw) {
        const int r = i / (kCw / 4), q = (i % (kCw / 4)) * 4;
        float* dk = sk + r * kCw + q;
        float* dv = sv + r * kCw + q;
        if (r < nrow && c0 + q < p.C) {               // C is a multiple of 4
            const int64_t off = (t0 + r) * p.C + c0 + q;
            cp_async16(dk, p.k + off);
            cp_async16(dv, p.v + off);
        } else {
            *reinterpret_cast<float4*>(dk) = make_float4(0.f, 0.f, 0.f, 0.f);
            *reinterpret_cast<float4*>(dv) = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    cp_async_commit();
    const float w = live ? p.w[c] : 0.f, u = live ? p.u[c] : 0.f;
    cp_async_wait_all();
    __syncthreads();

    // ---- pass 1: the tile's state from an empty start, resets at sequence starts
    int n = find_seq(p.cu, p.B, t0);
    int64_t nstart = p.cu[n], nend = p.cu[n + 1];
    St s = empty_state(), s0_last = empty_state();
    int64_t first_start = -1, last_start = -1;
    for (int r = 0; r < nrow; ++r) {
        const int64_t t = t0 + r;
        while (t >= nend && n + 1 < p.B) {
            ++n;
            nstart = p.cu[n];
            nend = p.cu[n + 1];
        }
        if (t == nstart) {
            if (first_start < 0) first_start = t;
            last_start = t;
            s0_last = live ? load_state(p.state_in, n, p.C, c) : empty_state();
            s = s0_last;
        }
        s = step(s, w, sk[r * kCw + tid], sv[r * kCw + tid]);
    }
    const bool reset = last_start >= 0;
    const size_t slot = size_t(tile) * kCw + tid;
    if (reset) put(p.incl, tiles, slot, s);           // end state known: no carry reaches it
    else put(p.agg, tiles, slot, s);
    __threadfence();
    __syncthreads();
    if (tid == 0) st_release(&p.flags[tile], reset ? 2 : 1);

    // ---- incoming state for rows before the first sequence start ----------------
    St s_in = empty_state();
    if (first_start != t0) {
        float R = 0.f;                                // carry map: x -> decay(x, R w) (+) L
        St L = empty_state();
        bool done = false;
        for (int pci = ci - 1; pci >= 0 && !done; --pci) {
            const int pidx = pci * p.n_cb + cb;
            if (tid == 0) {
                const int f = rows::wait_flag(&p.flags[pidx]);
                if (f == 0) s_fail = 1;
                s_flag = f;
            }
            __syncthreads();
            const int f = s_flag;
            if (s_fail) break;
            const size_t ps = size_t(pidx) * kCw + tid;
            if (f == 2) {
                s_in = add(decay(get(p.incl, tiles, ps), R * w), L);
                done = true;
            } else {
                const int prow = int(p.T - int64_t(pci) * kR < kR ? p.T - int64_t(pci) * kR : kR);
                L = add(decay(get(p.agg, tiles, ps), R * w), L);
                R += float(prow);
            }
            __syncthreads();                          // s_flag is reused
        }
        if (!done && !s_fail) s_in = L;               // no predecessor (malformed cu_seqlens)
    }
    if (!reset) {
        put(p.incl, tiles, slot, add(decay(s_in, float(nrow) * w), s));
        __threadfence();
        __syncthreads();
        if (tid == 0) st_release(&p.flags[tile], 2);
    }
    if (tid == 0 && s_fail) atomicAdd(&g_wkv_timeouts, 1);

    // ---- pass 2: outputs from the staged tile ------------------------------------
    if (!live) return;
    n = find_seq(p.cu, p.B, t0);
    nstart = p.cu[n];
    nend = p.cu[n + 1];
    s = s_in;
    for (int r = 0; r < nrow; ++r) {
        const int64_t t = t0 + r;
        while (t >= nend && n + 1 < p.B) {
            ++n;
            nstart = p.cu[n];
            nend = p.cu[n + 1];
        }
        if (t == nstart)   // the last start may continue past this tile: its state
                           // was read in pass 1 (state_out may alias state_in)
            s = t == last_start ? s0_last : load_state(p.state_in, n, p.C, c);
        const float kt = sk[r * kCw + tid], vt = sv[r * kCw + tid];
        p.wkv[t * p.C + c] = output(s, u, kt, vt);
        s = step(s, w, kt, vt);
        if (t == nend - 1) store_state(p.state_out, n, p.C, c, s);
    }
}

}  // namespace

size_t wkv_workspace_bytes(int C, int64_t T) {
    const int64_t tiles = ((T + kR - 1) / kR) * ((C + kCw - 1) / kCw);
    auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
    return up(sizeof(int)) + up(size_t(tiles) * sizeof(int)) + 2 * up(size_t(tiles) * kCw * 3 * sizeof(float));
}

void wkv_bind_workspace(WkvParams& p, void* ws) {
    auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
    char* w = static_cast<char*>(ws);
    p.n_cb = (p.C + kCw - 1) / kCw;
    p.n_tiles = int(((p.T + kR - 1) / kR) * p.n_cb);
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
        wkv_init_kernel<<<unsigned((init_items + 255) / 256), 256, 0, s>>>(p);
        timer_end(s);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    if (p.n_tiles == 0) return cudaSuccess;
    const int smem = 2 * kR * kCw * int(sizeof(float));
    cudaError_t e = ensure_smem(reinterpret_cast<const void*>(wkv_rows_kernel), smem);
    if (e != cudaSuccess) return e;
    timer_begin(s, "wkv_rows_kernel");
    wkv_rows_kernel<<<unsigned(p.n_tiles), kCw, smem, s>>>(p);
    timer_end(s);
    return cudaGetLastError();
}

int wkv_read_timeouts() {
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_wkv_timeouts, sizeof(int)) != cudaSuccess) return -1;
    return v;
}

}  // namespace gdn
