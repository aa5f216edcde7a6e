// Selective-scan rows: h_t = a_t h_{t-1} + b_t per channel over the rows of
// every sequence, from the incoming state h_in ("perf(mamba): prefill text
// prompts in multi-token chunks", Implementation, add_selective_scan_rows).
//
// The page scans the rows of one chunk by doubling rounds; here the whole
// prompt is one HBM-bound pass.  Tiles of 64 rows x 32 channels (16 KB, so
// that many CTAs per SM keep enough loads in flight) are taken in
// ticket order (a global counter), so every tile's predecessor in time is
// already running or done.  A CTA stages its tile in shared memory once
// (cp.async); each of its four warps reduces its 16 rows to the affine map
// h -> A h + B (as four interleaved chains of 4 rows, so that independent
// multiply-add chains hide the latency); warp 0 composes the tile's map,
// publishes it, finds the tile's incoming state by looking back over the
// predecessors' published maps and end states (decoupled look-back),
// publishes the tile's end state and hands every warp its incoming state;
// the warps then write h_t from the staged tile: a and b are read from HBM
// once and h written once.  A sequence start is folded into the staged row
// (a := 0, b := a h_in + b), so the map of a tile with a start ignores its
// input (its end state is published at once) and no state is read after
// the first pass, which keeps an aliased h_in / h_out safe.
#include "gdn_common.cuh"
#include "rows_common.cuh"
#include "tc_ptx.cuh"

namespace gdn {

__device__ int g_scan_timeouts = 0;   // bumped by a CTA whose bounded look-back ran out

namespace {

using namespace ptx;
using namespace rows;

constexpr int kRows = rows::kScanRows;            // rows of a tile
constexpr int kWarpRows = kRows / kWarps;          // rows of a warp
constexpr int kChainRows = kWarpRows / kChains;    // rows of one of a thread's chains

// Zero the ticket and the tile flags; end state of every empty sequence.
__global__ void scan_init_kernel(const ScanParams p) {
    ptx::griddep_wait();                              // the grid before may still use the flags
    const int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i == 0) *p.ticket = 0;
    if (i < p.n_tiles) p.flags[i] = 0;
    if (i < int64_t(p.B) * p.C) {
        const int n = int(i / p.C);
        if (p.cu[n + 1] <= p.cu[n]) p.h_out[i] = p.h_in ? p.h_in[i] : 0.f;
    }
}

__global__ void __launch_bounds__(kThreads) scan_rows_kernel(const ScanParams p) {
    griddep_wait();                                   // ticket and flags from scan_init_kernel
    extern __shared__ __align__(16) float sm_scan[];
    float* sa = sm_scan;                              // [kRows][kCols]
    float* sb = sm_scan + kRows * kCols;
    __shared__ int s_tile;
    __shared__ int s_seq[kRows], s_mark[kRows];
    __shared__ float s_A[kWarps][kCols], s_B[kWarps][kCols], s_in[kWarps][kCols];
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
    stage_tile<kRows>(sa, sb, p.a, p.b, t0, nrow, c0, p.C, tid);
    fill_row_info(p.cu, p.B, t0, nrow, tid, s_seq, s_mark);
    cp_async_wait_all();
    __syncthreads();

    // ---- pass 1: the map of the warp's rows, starts folded into the rows ------
    float A[kChains], Bv[kChains];
#pragma unroll
    for (int j = 0; j < kChains; ++j) {
        A[j] = 1.f;
        Bv[j] = 0.f;
    }
    int first = -1;
    const int rw = warp * kWarpRows;
#pragma unroll 4
    for (int i = 0; i < kChainRows; ++i) {
#pragma unroll
        for (int j = 0; j < kChains; ++j) {
            const int r = rw + j * kChainRows + i;
            if (r < nrow) {
                float ar = sa[r * kCols + lane], br = sb[r * kCols + lane];
                if (s_mark[r] & kRowStart) {
                    const float h0 = (live && p.h_in) ? p.h_in[int64_t(s_seq[r]) * p.C + c] : 0.f;
                    br = fmaf(ar, h0, br);
                    ar = 0.f;
                    sa[r * kCols + lane] = ar;
                    sb[r * kCols + lane] = br;
                    if (first < 0 || r < first) first = r;
                }
                A[j] = ar * A[j];
                Bv[j] = fmaf(ar, Bv[j], br);
            }
        }
    }
    {
        float Aw = A[0], Bw = Bv[0];
#pragma unroll
        for (int j = 1; j < kChains; ++j) {
            Bw = fmaf(A[j], Bw, Bv[j]);
            Aw = A[j] * Aw;
        }
        s_A[warp][lane] = Aw;
        s_B[warp][lane] = Bw;
        if (lane == 0) s_first[warp] = first;
    }
    __syncthreads();

    // ---- warp 0: publish, look back, hand out the warps' incoming states ------
    if (warp == 0) {
        float At = s_A[0][lane], Bt = s_B[0][lane];
        bool reset = s_first[0] >= 0;
#pragma unroll
        for (int w = 1; w < kWarps; ++w) {
            Bt = fmaf(s_A[w][lane], Bt, s_B[w][lane]);
            At = s_A[w][lane] * At;
            reset = reset || s_first[w] >= 0;
        }
        const size_t slot = size_t(tile) * kCols + lane;
        if (reset) {
            p.incl[slot] = Bt;                        // end state known: no carry reaches it
        } else {
            p.agg_a[slot] = At;
            p.agg_b[slot] = Bt;
        }
        __threadfence();
        __syncwarp();
        if (lane == 0) st_release(&p.flags[tile], reset ? 2 : 1);
        float h_in = 0.f;
        bool fail = false;
        if (s_first[0] != 0) {                        // row 0 continues the previous tile
            float ca = 1.f, cbv = 0.f;                // h_in = ca * (end state of pred) + cbv
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
                // L2 reads (__ldcg): another SM wrote these, and L1 is not coherent
                if (f == 2) {
                    h_in = fmaf(ca, __ldcg(p.incl + ps), cbv);
                    done = true;
                } else {
                    cbv = fmaf(ca, __ldcg(p.agg_b + ps), cbv);
                    ca *= __ldcg(p.agg_a + ps);
                }
            }
            if (!done && !fail) h_in = cbv;           // no predecessor (malformed cu_seqlens)
        }
        if (!reset) {
            p.incl[slot] = fmaf(At, h_in, Bt);
            __threadfence();
            __syncwarp();
            if (lane == 0) st_release(&p.flags[tile], 2);
        }
        if (fail && lane == 0) atomicAdd(&g_scan_timeouts, 1);
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            s_in[w][lane] = h_in;
            h_in = fmaf(s_A[w][lane], h_in, s_B[w][lane]);
        }
    }
    __syncthreads();

    // ---- pass 2: h_t from the staged rows, each chain from its own input -------
    if (!live) return;
    float h[kChains];
    h[0] = s_in[warp][lane];
#pragma unroll
    for (int j = 1; j < kChains; ++j) h[j] = fmaf(A[j - 1], h[j - 1], Bv[j - 1]);
#pragma unroll 4
    for (int i = 0; i < kChainRows; ++i) {
#pragma unroll
        for (int j = 0; j < kChains; ++j) {
            const int r = rw + j * kChainRows + i;
            if (r < nrow) {
                h[j] = fmaf(sa[r * kCols + lane], h[j], sb[r * kCols + lane]);
                p.h_rows[(t0 + r) * p.C + c] = h[j];
                if (s_mark[r] & kRowEnd) p.h_out[int64_t(s_seq[r]) * p.C + c] = h[j];
            }
        }
    }
}

}  // namespace

size_t scan_workspace_bytes(int C, int64_t T) {
    const int64_t n_cb = (C + rows::kCols - 1) / rows::kCols;
    const int64_t n_chunks = (T + rows::kScanRows - 1) / rows::kScanRows;
    const int64_t tiles = n_cb * n_chunks;
    auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
    return up(sizeof(int)) + up(size_t(tiles) * sizeof(int)) + 3 * up(size_t(tiles) * rows::kCols * sizeof(float));
}

void scan_bind_workspace(ScanParams& p, void* ws) {
    auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
    char* w = static_cast<char*>(ws);
    p.n_cb = (p.C + rows::kCols - 1) / rows::kCols;
    const int64_t n_chunks = (p.T + rows::kScanRows - 1) / rows::kScanRows;
    p.n_tiles = int(n_chunks * p.n_cb);
    p.ticket = reinterpret_cast<int*>(w);
    w += up(sizeof(int));
    p.flags = reinterpret_cast<int*>(w);
    w += up(size_t(p.n_tiles) * sizeof(int));
    const size_t vec = up(size_t(p.n_tiles) * rows::kCols * sizeof(float));
    p.agg_a = reinterpret_cast<float*>(w);
    p.agg_b = reinterpret_cast<float*>(w + vec);
    p.incl = reinterpret_cast<float*>(w + 2 * vec);
}

cudaError_t launch_scan_rows(const ScanParams& p, cudaStream_t s) {
    const int64_t init_items = int64_t(p.B) * p.C > p.n_tiles ? int64_t(p.B) * p.C : p.n_tiles;
    if (init_items > 0) {
        timer_begin(s, "scan_init_kernel");
        cudaError_t e = launch_pdl(scan_init_kernel, dim3(unsigned((init_items + 255) / 256)), 256, 0, s, p);
        timer_end(s);
        if (e != cudaSuccess) return e;
    }
    if (p.n_tiles == 0) return cudaSuccess;
    const int smem = 2 * rows::kScanRows * rows::kCols * int(sizeof(float));
    cudaError_t e = ensure_smem(reinterpret_cast<const void*>(scan_rows_kernel), smem);
    if (e != cudaSuccess) return e;
    timer_begin(s, "scan_rows_kernel");
    e = launch_pdl(scan_rows_kernel, dim3(unsigned(p.n_tiles)), rows::kThreads, unsigned(smem), s, p);
    timer_end(s);
    return e;
}

int scan_read_timeouts() {
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_scan_timeouts, sizeof(int)) != cudaSuccess) return -1;
    return v;
}

}  // namespace gdn
