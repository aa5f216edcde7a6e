// Internal declarations shared by the CUDA translation units of libgdn.so.
// Nothing here is part of the public ABI (include/gdn.h).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "gdn.h"

namespace gdn {

constexpr int kMaxChunk = 64;     // static padding of the triangular solve
constexpr int kNeumann = 8;       // diagonal block size of the Neumann stage

// Everything a chunk kernel needs.  Token strides are in elements so that q,
// k, v can be read from separate [T, H, d] tensors or from the [T, C]
// output of the short convolution.
// Segments of the segment-parallel scan that seg_out_kernel's group table
// covers (more use uniform groups).
constexpr int kSegTable = 64;

struct ChunkParams {
    const void* q;
    const void* k;
    const void* v;
    int64_t q_stride, k_stride, v_stride;  // elements between consecutive tokens
    const float* g;
    const float* beta;
    const float* state_in;
    float* state_out;
    void* out;
    const int32_t* cu;
    int64_t t_cap;  // tokens in the buffers (rows at or beyond it are never touched)
    int B, Hk, Hv, dk, dv, chunk;
    int l2norm;
    float eps;
    float q_scale;
    // Segment-parallel scan (tensor-core path only).  seg_phase 0: one pass
    // over every sequence.  Phase 1: segment 0 of each sequence in full, every
    // later segment s twice: from a zero state (its end state is the offset
    // B_s, its outputs O' go to `out`) and from the identity with V = 0 (its
    // end state is the transition M_s, its outputs, the output map G, go to
    // g_out).  seg_out_kernel then forms every segment's incoming state S_s
    // (S_{s+1} = M_s S_s + B_s), the outputs O = O' + G S_s of segments
    // s >= 1 and the final state.  seg_ws holds, per value head and segment
    // slot, three 128 x 128 fp32 matrices: B_s and S_s row-major [dk][dv], M_s
    // stored transposed (element (i, j) of M_s at j * dk + i); the slot of
    // (sequence n, segment s) is cu[n] / (seg_chunks * chunk) + n + s.  g_out
    // is bf16 laid out like `out`.
    int seg_chunks;
    int seg_phase;
    float* seg_ws;
    int64_t seg_slots;       // slots per value head
    int seg_max;             // most segments any sequence can have (grid size)
    int seg_groups;          // chunk groups per segment in seg_out_kernel, beyond the table
    int seg_final_cta;       // 1: a CTA of its own forms the final state; 0: the last group's
    // seg_out_kernel's CTAs per (sequence, value head) when seg_max - 1 <=
    // kSegTable: segment s >= 1 takes CTAs z with seg_gstart[s - 1] <= z <
    // seg_gstart[s] (seg_gstart[0] = 0), one chunk group each; the final
    // state's CTA, if any, is z = seg_gstart[seg_max - 1].  Later segments
    // (more state steps before their outputs) get more groups.
    int16_t seg_gstart[kSegTable + 1];
    void* g_out;
    // Split preparation (tensor-core path only).  When prep_ws is set, a
    // separate pass solves every chunk's S-independent part (inverse, U0, W,
    // the intra-chunk output weights P, the scaled queries) in parallel over
    // all chunks and stores one record per (value head, chunk slot); the
    // state pass then only streams the records.  The slot of chunk c of
    // sequence n is t0_n / chunk + n + c, with t0_n the sequence's clamped
    // first token.
    uint8_t* prep_ws;
    int64_t prep_slots;      // slots per value head
};

// Selective-scan rows (h_t = a_t h_{t-1} + b_t per channel).  a, b, h_rows
// [T, C] fp32, h_in / h_out [B, C]; the workspace holds the ticket counter,
// one flag per tile and the tiles' published maps and end states.
struct ScanParams {
    const float* a;
    const float* b;
    const float* h_in;       // or nullptr (zero state)
    float* h_out;
    float* h_rows;
    const int32_t* cu;
    int64_t T;
    int B, C;
    int n_cb, n_tiles;       // channel blocks; tiles (time chunks x channel blocks)
    int* ticket;
    int* flags;              // per tile: 0 none, 1 map published, 2 end state published
    float* agg_a;            // per tile and channel: the map h -> A h + B of its rows
    float* agg_b;
    float* incl;             // per tile and channel: the state after its last row
};
size_t scan_workspace_bytes(int C, int64_t T);
void scan_bind_workspace(ScanParams& p, void* ws);
cudaError_t launch_scan_rows(const ScanParams& p, cudaStream_t s);
int scan_read_timeouts();   // bounded waits of the scan that ran out (-1 on a CUDA error)

// RWKV-4 WKV rows.  k, v, wkv [T, C] fp32; w, u [C]; state_in / state_out
// [B, 3, C] holding num, den, max.  Same ticket / flag workspace as the scan;
// agg and incl hold (num, den, max) per tile and channel, each component a
// block of n_tiles * 128 floats.
struct WkvParams {
    const float* k;
    const float* v;
    const float* w;
    const float* u;
    const float* state_in;   // or nullptr (empty state (0, 0, -1e38))
    float* state_out;
    float* wkv;
    const int32_t* cu;
    int64_t T;
    int B, C;
    int n_cb, n_tiles;
    int* ticket;
    int* flags;
    float* agg;              // per tile: the state its rows build from an empty start
    float* incl;             // per tile: the state after its last row
};
size_t wkv_workspace_bytes(int C, int64_t T);
void wkv_bind_workspace(WkvParams& p, void* ws);
cudaError_t launch_wkv_rows(const WkvParams& p, cudaStream_t s);
int wkv_read_timeouts();
int tc_read_timeouts();     // same for the tensor-core chunk kernel

// Full-attention rows over a KV cache plus the chunk's causal prefix: q
// [T, Hq, 128], k, v [T, Hkv, 128], caches [B, Hkv, cap, 128], o [T, Hq, 128],
// all bf16; cache_len [B] int32 (device).
struct AttnParams {
    const void* q;
    const void* k;
    const void* v;
    void* k_cache;
    void* v_cache;
    void* o;
    const int32_t* cu;
    const int32_t* cache_len;
    int64_t T;
    int64_t max_len;         // upper bound on any sequence's length (grid size)
    int B, Hq, Hkv, cap;
    float scale;
};
cudaError_t launch_attn_rows(const AttnParams& p, cudaStream_t s);
int attn_read_timeouts();

// Raise a kernel's dynamic shared-memory limit to at least `bytes` on the
// current device; the attribute is set once per (device, kernel, size) rather
// than on every launch.
cudaError_t ensure_smem(const void* kernel, int bytes);

// The part of gdn_workspace_bytes a prefill cannot run without (the short
// convolution's output); the segment maps and chunk records are optional.
size_t prefill_required_workspace(const gdn_prefill_desc* d);

// Launch as a programmatic dependent of the preceding grid in the stream: the
// kernel's own griddep_wait() orders it after that grid, while its launch and
// set-up overlap the end of it (its CTAs start on the SMs the preceding grid
// has left).
template <typename... Kargs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(Kargs...), dim3 grid, unsigned block, unsigned smem, cudaStream_t s,
                       Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Launch timing: bracket a kernel launch with timer_begin / timer_end on the
// launch stream (no-ops unless gdn_launch_timer_start turned recording on).
void timer_begin(cudaStream_t s, const char* kernel);
void timer_end(cudaStream_t s);

// Bytes of one chunk record of the split preparation.
constexpr size_t kPrepRecordBytes = 82432;

struct ConvParams {
    const void* x;           // [T, C]
    const float* w;          // [C, K]
    const float* state_in;   // [B, C, K-1] or nullptr
    float* state_out;        // [B, C, K-1] or nullptr
    void* y;                 // [T, C] (workspace), same dtype as x
    const int32_t* cu;
    int64_t T;
    int B, C, K, act;
};

struct StepParams {
    const void* q;
    const void* k;
    const void* v;
    const void* conv_x;      // [B, C] or nullptr
    const float* conv_w;
    const float* conv_state_in;
    float* conv_state_out;
    int conv_K, conv_act;
    const float* g;
    const float* beta;
    const float* state_in;
    float* state_out;
    void* out;
    int B, Hk, Hv, dk, dv;
    int l2norm;
    float eps;
    float q_scale;
};

// Launchers (return cudaSuccess or the launch error).
cudaError_t launch_chunk_simt(const ChunkParams& p, int dtype, cudaStream_t s);
cudaError_t launch_conv(const ConvParams& p, int dtype, cudaStream_t s);
cudaError_t launch_conv_state(const ConvParams& p, int dtype, cudaStream_t s);
cudaError_t launch_step(const StepParams& p, int dtype, cudaStream_t s);
cudaError_t launch_step_conv_state(const StepParams& p, int dtype, cudaStream_t s);

// ---- small device helpers --------------------------------------------------

__device__ __forceinline__ float load_elem(const float* p, int64_t i) { return p[i]; }
__device__ __forceinline__ float load_elem(const __nv_bfloat16* p, int64_t i) {
    return __bfloat162float(p[i]);
}
__device__ __forceinline__ void store_elem(float* p, int64_t i, float x) { p[i] = x; }
__device__ __forceinline__ void store_elem(__nv_bfloat16* p, int64_t i, float x) {
    p[i] = __float2bfloat16_rn(x);
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

}  // namespace gdn
