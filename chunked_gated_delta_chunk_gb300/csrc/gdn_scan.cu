// Selective-scan rows: h_t = a_t h_{t-1} + b_t per channel over the rows of
// every sequence, from the incoming state h_in ("perf(mamba): prefill text
// prompts in multi-token chunks", Implementation, add_selective_scan_rows).
//
// The page scans the rows of one chunk by doubling rounds; here the whole
// prompt is one HBM-bound pass.  Tiles of kScanRows rows x kScanCols channels
// are taken in ticket order (a global counter), so every tile's predecessor
// in time is already running or done.  A CTA stages its tile in shared memory
// once (cp.async), reduces it to the affine map h -> A h + B of its rows,
// publishes that map, finds its incoming state by looking back over the
// predecessors' published maps and end states (decoupled look-back), publishes
// its own end state, and writes h_t for its rows from the staged tile: a and
// b are read from HBM once and h written once.  A sequence start inside a
// tile resets the map (A = 0, B = h_in), so such a tile needs no look-back.
#include "gdn_common.cuh"
#include "rows_common.cuh"
#include "tc_ptx.cuh"

namespace gdn {

__device__ int g_scan_timeouts = 0;   // bumped by a CTA whose bounded look-back ran out

namespace {

using namespace ptx;

constexpr int kScanRows = rows::kRows;
constexpr int kScanCols = rows::kCols;        // one thread per channel
using rows::find_seq;
using rows::st_release;

// Zero the ticket and the tile flags; end state of every empty sequence.
__global__ void scan_init_kernel(const ScanParams p) {
    const int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i == 0) *p.ticket = 0;
    if (i < p.n_tiles) p.flags[i] = 0;
    if (i < int64_t(p.B) * p.C) {
        const int n = int(i / p.C);
        if (p.cu[n + 1] <= p.cu[n]) p.h_out[i] = p.h_in ? p.h_in[i] : 0.f;
    }
}

__global__ void __launch_bounds__(kScanCols) scan_rows_kernel(const ScanParams p) {
    extern __shared__ __align__(16) float sm_scan[];
    float* sa = sm_scan;                              // [kScanRows][kScanCols]
    float* sb = sm_scan + kScanRows * kScanCols;
    __shared__ int s_tile, s_flag, s_fail;
    const int tid = threadIdx.x;
    if (tid == 0) {
        s_tile = atomicAdd(p.ticket, 1);
        s_fail = 0;
    }
    __syncthreads();
    const int tile = s_tile;
    const int ci = tile / p.n_cb, cb = tile % p.n_cb;
    const int64_t t0 = int64_t(ci) * kScanRows;
    const int nrow = int(p.T - t0 < kScanRows ? p.T - t0 : kScanRows);
    const int c0 = cb * kScanCols;
    const int c = c0 + tid;
    const bool live = c < p.C;

    // ---- stage the tile: 16-byte copies, 32 threads per row -----------------
    for (int i = tid; i < kScanRows * (kScanCols / 4); i += kScanCols) {
        const int r = i / (kScanCols / 4), q = (i % (kScanCols / 4)) * 4;
        float* da = sa + r * kScanCols + q;
        float* db = sb + r * kScanCols + q;
        if (r < nrow && c0 + q < p.C) {               // C is a multiple of 4
            const int64_t off = (t0 + r) * p.C + c0 + q;
            cp_async16(da, p.a + off);
            cp_async16(db, p.b + off);
        } else {
            *reinterpret_cast<float4*>(da) = make_float4(0.f, 0.f, 0.f, 0.f);
            *reinterpret_cast<float4*>(db) = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    cp_async_commit();
    cp_async_wait_all();
    __syncthreads();

    // ---- pass 1: the tile's affine map, resets at sequence starts -----------
    int n = find_seq(p.cu, p.B, t0);
    int64_t nstart = p.cu[n], nend = p.cu[n + 1];
    float A = 1.f, Bv = 0.f, h0_last = 0.f;
    int64_t first_start = -1, last_start = -1;       // first and last sequence start in the tile
    bool reset = false;
    for (int r = 0; r < nrow; ++r) {
        const int64_t t = t0 + r;
        while (t >= nend && n + 1 < p.B) {           // skip ended and empty sequences
            ++n;
            nstart = p.cu[n];
            nend = p.cu[n + 1];
        }
        if (t == nstart) {
            reset = true;
            if (first_start < 0) first_start = t;
            last_start = t;
            h0_last = (live && p.h_in) ? p.h_in[int64_t(n) * p.C + c] : 0.f;
            A = 0.f;
            Bv = h0_last;
        }
        const float ar = sa[r * kScanCols + tid], br = sb[r * kScanCols + tid];
        A = ar * A;
        Bv = fmaf(ar, Bv, br);
    }
    const size_t slot = size_t(tile) * kScanCols + tid;
    const int flag_idx = ci * p.n_cb + cb;
    // The tile's end state needs no carry once a sequence starts in it: publish
    // it at once.  Otherwise publish the map, and the end state after the
    // look-back.
    if (reset) {
        p.incl[slot] = Bv;
    } else {
        p.agg_a[slot] = A;
        p.agg_b[slot] = Bv;
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) st_release(&p.flags[flag_idx], reset ? 2 : 1);

    // ---- incoming state: rows before the tile's first sequence start need the
    // state after the previous tile (look back over the predecessors)
    float s_in = 0.f;
    const bool first_is_start = last_start >= 0 && first_start == t0;
    if (!first_is_start) {
        float ca = 1.f, cbv = 0.f;                    // s_in = ca * (end state of pred) + cbv
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
            const size_t ps = size_t(pidx) * kScanCols + tid;   // tile index of (pci, cb)
            // L2 reads (__ldcg): another SM wrote these, and L1 is not coherent
            if (f == 2) {
                s_in = fmaf(ca, __ldcg(p.incl + ps), cbv);
                done = true;
            } else {
                cbv = fmaf(ca, __ldcg(p.agg_b + ps), cbv);
                ca *= __ldcg(p.agg_a + ps);
            }
            __syncthreads();                          // s_flag is reused
        }
        if (!done && !s_fail) s_in = cbv;             // no predecessor (malformed cu_seqlens)
    }
    if (!reset) {
        p.incl[slot] = fmaf(A, s_in, Bv);
        __threadfence();
        __syncthreads();
        if (tid == 0) st_release(&p.flags[flag_idx], 2);
    }
    if (tid == 0 && s_fail) atomicAdd(&g_scan_timeouts, 1);

    // ---- pass 2: h_t from the staged tile ------------------------------------
    if (!live) return;
    n = find_seq(p.cu, p.B, t0);
    nstart = p.cu[n];
    nend = p.cu[n + 1];
    float h = s_in;
    for (int r = 0; r < nrow; ++r) {
        const int64_t t = t0 + r;
        while (t >= nend && n + 1 < p.B) {
            ++n;
            nstart = p.cu[n];
            nend = p.cu[n + 1];
        }
        if (t == nstart)   // the last start may continue past this tile: its state
                           // was read in pass 1 (h_out may alias h_in)
            h = t == last_start ? h0_last : (p.h_in ? p.h_in[int64_t(n) * p.C + c] : 0.f);
        h = fmaf(sa[r * kScanCols + tid], h, sb[r * kScanCols + tid]);
        p.h_rows[t * p.C + c] = h;
        if (t == nend - 1) p.h_out[int64_t(n) * p.C + c] = h;
    }
}

}  // namespace

size_t scan_workspace_bytes(int C, int64_t T) {
    const int64_t n_cb = (C + kScanCols - 1) / kScanCols;
    const int64_t n_chunks = (T + kScanRows - 1) / kScanRows;
    const int64_t tiles = n_cb * n_chunks;
    auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
    return up(sizeof(int)) + up(size_t(tiles) * sizeof(int)) + 3 * up(size_t(tiles) * kScanCols * sizeof(float));
}

void scan_bind_workspace(ScanParams& p, void* ws) {
    auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
    char* w = static_cast<char*>(ws);
    p.n_cb = (p.C + kScanCols - 1) / kScanCols;
    const int64_t n_chunks = (p.T + kScanRows - 1) / kScanRows;
    p.n_tiles = int(n_chunks * p.n_cb);
    p.ticket = reinterpret_cast<int*>(w);
    w += up(sizeof(int));
    p.flags = reinterpret_cast<int*>(w);
    w += up(size_t(p.n_tiles) * sizeof(int));
    const size_t vec = up(size_t(p.n_tiles) * kScanCols * sizeof(float));
    p.agg_a = reinterpret_cast<float*>(w);
    p.agg_b = reinterpret_cast<float*>(w + vec);
    p.incl = reinterpret_cast<float*>(w + 2 * vec);
}

cudaError_t launch_scan_rows(const ScanParams& p, cudaStream_t s) {
    const int64_t init_items = int64_t(p.B) * p.C > p.n_tiles ? int64_t(p.B) * p.C : p.n_tiles;
    if (init_items > 0) {
        timer_begin(s, "scan_init_kernel");
        scan_init_kernel<<<unsigned((init_items + 255) / 256), 256, 0, s>>>(p);
        timer_end(s);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    if (p.n_tiles == 0) return cudaSuccess;
    const int smem = 2 * kScanRows * kScanCols * int(sizeof(float));
    cudaError_t e = ensure_smem(reinterpret_cast<const void*>(scan_rows_kernel), smem);
    if (e != cudaSuccess) return e;
    timer_begin(s, "scan_rows_kernel");
    scan_rows_kernel<<<unsigned(p.n_tiles), kScanCols, smem, s>>>(p);
    timer_end(s);
    return cudaGetLastError();
}

int scan_read_timeouts() {
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_scan_timeouts, sizeof(int)) != cudaSuccess) return -1;
    return v;
}

}  // namespace gdn
